// prefill.cu -- the non-absorbed projection of the cached latent:
//   Y[t][n] = sLc_t * sum_{d<512} dec(Lc_t[d]) * W_UKV[d][n]      (bf16 out)
// and, optionally, the token's rope key dequantized, K_rope[t][j] = sRc_t * dec(Rc_t[j])
// (f32, one rounding of the exact product).
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
// description: the projection path dequantizes the cached Lc rows (value times
// the row's scale) before the kv_b up-projection.
//
// A dense contraction on the tensor cores (tcgen05, kind::f16 with bf16
// operands, f32 accumulators in TMEM), run by CTA pairs: one MMA of M = 256
// tokens x N = 256 columns x K = 16 spans the two SMs of a pair (cta_group::2),
// each SM holding 128 of the tokens (A, and the accumulator rows) and 128 of the
// columns (its half of the W stage), so each SM streams half of W per pair tile.
// The row scale sLc factors out of each output row, so A holds the e4m3 codes
// converted to bf16 (exact) and the epilogue multiplies by sLc.  The (pair
// token tile, column tile) units are numbered token-tile-major and every pair
// takes a contiguous range, converting its 256 tokens' A once (128 KB of shared
// memory per SM) and streaming W through a 4-stage TMA ring.
//
// Warp roles (12 warps per CTA):
//   warp 0 of CTA 0   issues the pair MMAs (whole warp, one elected lane); the
//                     commits arrive on the barriers of both CTAs.  TMEM (two
//                     256-column accumulators, so a tile's epilogue overlaps the
//                     next tile's MMAs) is allocated by warp 0 of both CTAs.
//   warp 1            TMA producer of this CTA's half of each W stage: [64 k-rows
//                     x 128 columns] as two [64 x 64] boxes (128-byte swizzle),
//                     an MN-major B operand; both halves complete on CTA 0's
//                     stage barrier.
//   warps 4-11        convert this CTA's 128 tokens to bf16 (K-major, 128-byte
//                     swizzle, one [128 x 64] chunk per warp) as soon as the MMAs
//                     of the previous token tile are done, then run the epilogue:
//                     warp w reads TMEM lanes 32 (w % 4) .. +31 (its token rows)
//                     and column half (w - 4) / 4, scales by sLc, rounds to bf16
//                     into a 4 KB shared-memory box and writes it with a TMA
//                     store (rows past T are clipped by the tensor map).  The CTA
//                     that converts a token tile for its first column tile also
//                     writes the tile's K_rope rows.
// Every wait is bounded (2 s); on a timeout the CTA sets the error word (if
// given), drains its MMAs, TMA loads and stores, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

using namespace ptx;

constexpr int PT_M = 128, PT_N = 256, PT_K = 512;
constexpr int KS = 64;                          // k-rows per W stage
constexpr int NST = 4;                          // W stages (each CTA: its half of the columns)
constexpr int NCONV = 8;                        // convert + epilogue warps
constexpr int WARP_CONV = 4;
constexpr int NTHREADS = (WARP_CONV + NCONV) * 32;
constexpr int ACHUNK = PT_M * 64 * 2;           // 16 KB: 128 rows x 64 bf16
constexpr int WBOX = KS * 64 * 2;               // 8 KB: 64 k-rows x 64 columns
constexpr int STAGE = 2 * WBOX;                 // 16 KB per CTA
constexpr int OBOX = 32 * 64 * 2;               // 4 KB: 32 rows x 64 columns of Y
constexpr int OFF_A = 0;
constexpr int OFF_B = 8 * ACHUNK;               // 128 KB
constexpr int OFF_O = OFF_B + NST * STAGE;      // 192 KB
constexpr int OFF_BAR = OFF_O + NCONV * OBOX;   // 224 KB
constexpr int SMEM = OFF_BAR + 256 + 1024;
constexpr int B_AREADY = 0, B_AFREE = 1, B_FULL = 2, B_EMPTY = B_FULL + NST,
              B_ACCF = B_EMPTY + NST, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2, NBAR = B_DRAIN + 1;
static_assert(NBAR * 8 + 16 <= 256, "barrier area");
static_assert(SMEM <= 232448, "shared memory per CTA");
constexpr uint64_t WAIT_NS = 2000000000ull;

// kind::f16 instruction descriptor with bf16 A and B (format 1), f32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f16(M, N, a_mn, b_mn) | (1u << 7) | (1u << 10);
}

__device__ __forceinline__ void sts128p(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// two e4m3 bytes -> bf16x2 (exact: every e4m3 value is a bf16 value)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  const uint32_t h = e4m3x2_to_f16x2(v);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
  return r;
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int PM = 2 * PT_M;   // tokens per pair tile

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
prefill_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
               const int64_t* __restrict__ slots, int64_t n_slots, int64_t T, int N,
               float* __restrict__ k_rope, unsigned* __restrict__ err,
               const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap ymap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + NBAR * 8 + 4);

  // this pair's range of (pair token tile, column tile) units; both CTAs take the same range
  const int64_t MP = (T + PM - 1) / PM, NT = N / PT_N, tot = MP * NT;
  const int64_t npair = gridDim.x / 2, pid = blockIdx.x / 2;
  const int64_t f0 = tot * pid / npair, f1 = tot * (pid + 1) / npair;
  if (f0 >= f1) return;   // same for both CTAs of the pair

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_AREADY], 2 * NCONV);
    mbar_init(&bars[B_AFREE], 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bars[B_FULL + s], 1);
      mbar_init(&bars[B_EMPTY + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_ACCF + b], 1);
      mbar_init(&bars[B_ACCE + b], 2 * NCONV);
    }
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = smem_u32(sm + OFF_A), b_base = smem_u32(sm + OFF_B);
  auto leader_bar = [&](int i) { return map_to(smem_u32(&bars[i]), 0); };
  auto fail = [&]() {
    *abort_flag = 1;
    if (err != nullptr) atomicOr(err, ERR_TIMEOUT);
  };

  if (warp == 0 && leader) {
    // ---------------------------------------------------------- pair MMA issuer
    const uint32_t id = idesc_bf16(2 * PT_M, PT_N, false, true);
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_cluster(bar, par, abort_flag, WAIT_NS));
    };
    bool ok = true;
    int64_t g = 0;
    int seg = 0;
    for (int64_t f = f0, u = 0; ok && f < f1; ++f, ++u) {
      const bool first = (f == f0) || (f % NT == 0);
      if (first) {
        ok = wait(&bars[B_AREADY], seg & 1);
        ++seg;
        if (!ok) break;
      }
      const int buf = (int)(u & 1);
      if (!wait(&bars[B_ACCE + buf], (uint32_t)((u >> 1) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem + buf * PT_N;
      for (int ks = 0; ks < PT_K / KS; ++ks, ++g) {
        const int st = (int)(g % NST);
        if (!wait(&bars[B_FULL + st], (uint32_t)((g / NST) & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KS / 16; ++kk) {
          const int k16 = ks * (KS / 16) + kk;
          const uint64_t ad = smem_desc(a_base + (k16 >> 2) * ACHUNK + (k16 & 3) * 32, 16, 1024, SW128);
          const uint64_t bd = smem_desc(b_base + st * STAGE + kk * 2048, WBOX, 1024, SW128);
          mma_f16_pair_warp(d, ad, bd, id, (ks | kk) != 0);
        }
        mma_commit_pair_warp(&bars[B_EMPTY + st], 3);
      }
      if (!ok) break;
      mma_commit_pair_warp(&bars[B_ACCF + buf], 3);
      const bool last = (f + 1 == f1) || ((f + 1) % NT == 0);
      if (last) mma_commit_pair_warp(&bars[B_AFREE], 3);
    }
    if (!ok && lane == 0) fail();
    const int zero = 0;
    mma_commit_pair_warp(&bars[B_DRAIN], 1);
    (void)mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- W producer (this CTA's column half)
    bool ok = true;
    int64_t g = 0;
    const uint64_t keep = l2_policy_evict_last();
    for (int64_t f = f0; ok && f < f1; ++f) {
      const int x0 = (int)(f % NT) * PT_N + (int)rank * (PT_N / 2);
      for (int ks = 0; ks < PT_K / KS; ++ks, ++g) {
        const int st = (int)(g % NST);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_EMPTY + st],
                                               (uint32_t)((g / NST) & 1) ^ 1, abort_flag, WAIT_NS));
        if (!ok) break;
        if (lane == 0) {
          // the leader's FULL barrier expects both halves; W stays in L2 for the
          // other token tiles (Y, streamed out, goes first)
          if (leader) mbar_arrive_expect_tx(&bars[B_FULL + st], 2 * STAGE);
          const uint32_t fb = leader_bar(B_FULL + st);
          const uint32_t dst = b_base + st * STAGE;
#pragma unroll
          for (int a2 = 0; a2 < 2; ++a2)
            tma_load_2d_pair_hint(dst + a2 * WBOX, &wmap, x0 + 64 * a2, KS * ks, fb, keep);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) fail();
    if (leader) {
      // let the requested loads (both halves) land before the pair can exit
      const int zero = 0;
      for (int64_t gg = (g > NST ? g - NST : 0); gg < g; ++gg)
        (void)mbar_wait(&bars[B_FULL + (int)(gg % NST)], (uint32_t)((gg / NST) & 1), &zero,
                        WAIT_NS);
    }
    __syncwarp();
  } else if (warp >= WARP_CONV) {
    // ---------------------------------------------------------- convert + epilogue (own 128 rows)
    const int cw = warp - WARP_CONV;
    const int q = warp & 3;
    const int half = cw >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const uint32_t obox = smem_u32(sm + OFF_O + cw * OBOX);
    const int rin = lane >> 2, sub = lane & 3;
    const uint32_t aready = leader_bar(B_AREADY);
    const int64_t rbase = (int64_t)rank * PT_M;

    auto convert = [&](int64_t m, bool rope) {
      const uint32_t chunk = a_base + cw * ACHUNK;
      uint4 x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int64_t t = m * PM + rbase + 8 * i + rin;
        x[i] = make_uint4(0u, 0u, 0u, 0u);
        if (t < T) {
          const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
          if (slot >= 0 && slot < n_slots)
            x[i] = __ldg(reinterpret_cast<const uint4*>(codes + slot * D + cw * 64 + sub * 16));
          else if (err != nullptr && cw == 0)
            atomicOr(err, ERR_BLOCK_TABLE);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t h[8];
        h[0] = e4m3x2_to_bf16x2((uint16_t)(x[i].x & 0xFFFFu)); h[1] = e4m3x2_to_bf16x2((uint16_t)(x[i].x >> 16));
        h[2] = e4m3x2_to_bf16x2((uint16_t)(x[i].y & 0xFFFFu)); h[3] = e4m3x2_to_bf16x2((uint16_t)(x[i].y >> 16));
        h[4] = e4m3x2_to_bf16x2((uint16_t)(x[i].z & 0xFFFFu)); h[5] = e4m3x2_to_bf16x2((uint16_t)(x[i].z >> 16));
        h[6] = e4m3x2_to_bf16x2((uint16_t)(x[i].w & 0xFFFFu)); h[7] = e4m3x2_to_bf16x2((uint16_t)(x[i].w >> 16));
        const uint32_t o0 = (uint32_t)(i * 1024 + rin * 128 + (((2 * sub) ^ rin) << 4));
        const uint32_t o1 = (uint32_t)(i * 1024 + rin * 128 + (((2 * sub + 1) ^ rin) << 4));
        sts128p(chunk + o0, make_uint4(h[0], h[1], h[2], h[3]));
        sts128p(chunk + o1, make_uint4(h[4], h[5], h[6], h[7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive_cluster(aready);
      if (rope && k_rope != nullptr) {
        const int part = lane & 7;
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          const int64_t t = m * PM + rbase + cw * 16 + 4 * i + (lane >> 3);
          if (t >= T) break;
          const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
          float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (slot >= 0 && slot < n_slots) {
            const uint2 c8 = __ldg(reinterpret_cast<const uint2*>(codes + slot * D + DL + part * 8));
            const float sR = __ldg(&scales[slot * 2 + 1]);
            e4m3x4_to_f32(c8.x, v);
            e4m3x4_to_f32(c8.y, v + 4);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] *= sR;
          }
          float4* dst = reinterpret_cast<float4*>(k_rope + t * DR + part * 8);
          dst[0] = make_float4(v[0], v[1], v[2], v[3]);
          dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
      }
    };

    bool ok = true;
    int seg = 1;
    const uint32_t acce0 = leader_bar(B_ACCE), acce1 = leader_bar(B_ACCE + 1);
    const uint64_t stream_out = l2_policy_evict_first();
    convert(f0 / NT, f0 % NT == 0);
    for (int64_t f = f0, u = 0; f < f1; ++f, ++u) {
      const int64_t m = f / NT;
      const int buf = (int)(u & 1);
      ok = mbar_wait_warp(&bars[B_ACCF + buf], (uint32_t)((u >> 1) & 1), abort_flag, WAIT_NS);
      if (!ok) break;
      tc_fence_after();
      if (f + 1 < f1 && (f + 1) % NT == 0) {
        ok = mbar_wait_warp(&bars[B_AFREE], (uint32_t)((seg - 1) & 1), abort_flag, WAIT_NS);
        if (!ok) break;
        convert(m + 1, true);
        ++seg;
      }
      const int64_t t = m * PM + rbase + row;
      float sL = 0.f;
      if (t < T) {
        const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
        if (slot >= 0 && slot < n_slots) sL = __ldg(&scales[slot * 2]);
      }
      const int xcol = (int)(f % NT) * PT_N + half * 128;
#pragma unroll 1
      for (int sc = 0; sc < 2; ++sc) {
        uint32_t v[4][16];
        const uint32_t ta = tmem + lane_addr + buf * PT_N + half * 128 + sc * 64;
        tmem_ld16(ta, v[0]);
        tmem_ld16(ta + 16, v[1]);
        tmem_ld16(ta + 32, v[2]);
        tmem_ld16(ta + 48, v[3]);
        tmem_wait_ld();
        if (sc == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_cluster(buf ? acce1 : acce0);
        }
        uint32_t p[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            p[j * 8 + e] = f32x2_to_bf16x2(__uint_as_float(v[j][2 * e]) * sL,
                                          __uint_as_float(v[j][2 * e + 1]) * sL);
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          sts128p(obox + lane * 128 + ((c ^ (lane & 7)) << 4),
                  make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d_hint(&ymap, obox, xcol + sc * 64, (int)(m * PM + rbase + q * 32), stream_out);
          bulk_commit();
        }
      }
    }
    if (!ok && lane == 0) fail();
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  // warps 2 and 3, and warp 0 of the second CTA, have no role
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}

// 2-D bf16 map over a row-major [rows][cols] array: boxes of box_rows x 64
// columns, 128-byte swizzle.
cudaError_t make_map(const uint16_t* base, int64_t cols, int64_t rows, int box_rows,
                     CUtensorMap* map) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(base),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const uint8_t* codes, const float* scales, const int64_t* slots,
                           int64_t n_slots, int64_t T, const uint16_t* w, int N, uint16_t* y,
                           float* k_rope, unsigned* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // pairs that can be resident at once: the work is cut into that many ranges
  static std::atomic<int> memo[MAX_DEVICES];
  int max_pairs = 0;
  cudaError_t e = per_device(memo, [](int* v) {
    cudaError_t r = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (r != cudaSuccess) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NUM_SMS, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    int n = 0;
    r = cudaOccupancyMaxActiveClusters(&n, prefill_kernel, &cfg);
    *v = n < 1 ? 1 : (n > NUM_SMS / 2 ? NUM_SMS / 2 : n);
    return r;
  }, &max_pairs);
  if (e != cudaSuccess) return e;
  CUtensorMap wmap, ymap;
  e = make_map(w, N, PT_K, KS, &wmap);
  if (e != cudaSuccess) return e;
  e = make_map(y, N, T, 32, &ymap);
  if (e != cudaSuccess) return e;
  const int64_t tot = ((T + 2 * PT_M - 1) / (2 * PT_M)) * (N / PT_N);
  const int pairs = (int)(tot < max_pairs ? tot : max_pairs);
  const int grid = 2 * pairs;
  prefill_kernel<<<grid, NTHREADS, SMEM, s>>>(codes, scales, slots, n_slots, T, N, k_rope, err,
                                              wmap, ymap);
  return cudaGetLastError();
}

}  // namespace kv8
