// prefill.cu -- the non-absorbed projection of the cached latent:
//   Y[t][n] = sLc_t * sum_{d<512} dec(Lc_t[d]) * W_UKV[d][n]      (bf16 out)
// and, optionally, the token's rope key dequantized, K_rope[t][j] = sRc_t * dec(Rc_t[j])
// (f32, one rounding of the exact product).
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
// description: the projection path dequantizes the cached Lc rows (value times
// the row's scale) before the kv_b up-projection.
//
// A dense contraction on the tensor cores (tcgen05, kind::f16 with bf16
// operands, f32 accumulators in TMEM).  Tiles of 128 tokens x 256 columns,
// K = 512.  The row scale sLc factors out of each output row, so A holds the
// e4m3 codes converted to bf16 (exact) and the epilogue multiplies by sLc.
// The (token tile, column tile) pairs are numbered token-tile-major and every
// CTA takes a contiguous range, converting a token tile's A once (128 KB of
// shared memory) and streaming W through a 3-stage TMA ring.
//
// Warp roles (8 warps):
//   warp 0      issues the MMAs (whole warp, one elected lane); owns TMEM
//               (two 256-column accumulators, so a tile's epilogue overlaps
//               the next tile's MMAs).
//   warp 1      TMA producer of the W stages: [64 k-rows x 256 columns] as four
//               [64 x 64] boxes (128-byte swizzle), read by the MMA as an
//               MN-major B operand.
//   warps 4-7   convert the token tile's codes to bf16 (K-major, 128-byte
//               swizzle, eight [128 x 64] chunks) at the start of each token
//               tile, then run the epilogue: thread = token row = TMEM lane;
//               TMEM -> x sLc -> bf16 -> 16-byte stores.  The CTA that holds a
//               token tile's first column tile also writes its K_rope rows.
// Every wait is bounded (2 s); on a timeout the CTA sets the error word (if
// given), drains its MMAs and TMA loads, frees TMEM and exits.
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
constexpr int NST = 3;                          // W stages
constexpr int ACHUNK = PT_M * 64 * 2;           // 16 KB: 128 rows x 64 bf16
constexpr int STAGE = 64 * PT_N * 2;            // 32 KB: 64 k-rows x 256 columns
constexpr int OFF_A = 0;
constexpr int OFF_B = 8 * ACHUNK;               // 128 KB
constexpr int OFF_BAR = OFF_B + NST * STAGE;    // 224 KB
constexpr int SMEM = OFF_BAR + 256 + 1024;
constexpr int B_AREADY = 0, B_AFREE = 1, B_FULL = 2, B_EMPTY = B_FULL + NST,
              B_ACCF = B_EMPTY + NST, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2, NBAR = B_DRAIN + 1;
static_assert(NBAR * 8 + 16 <= 256, "barrier area");
constexpr uint64_t WAIT_NS = 2000000000ull;

// kind::f16 instruction descriptor with bf16 A and B (format 1), f32 D.
constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
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

__global__ void __launch_bounds__(256, 1)
prefill_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
               const int64_t* __restrict__ slots, int64_t n_slots, int64_t T, int N,
               uint16_t* __restrict__ y, float* __restrict__ k_rope, unsigned* __restrict__ err,
               const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + NBAR * 8 + 4);

  // this CTA's range of (token tile, column tile) pairs
  const int64_t MT = (T + PT_M - 1) / PT_M, NT = N / PT_N, tot = MT * NT;
  const int64_t f0 = tot * blockIdx.x / gridDim.x, f1 = tot * (blockIdx.x + 1) / gridDim.x;
  if (f0 >= f1) return;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_AREADY], 4);
    mbar_init(&bars[B_AFREE], 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bars[B_FULL + s], 1);
      mbar_init(&bars[B_EMPTY + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_ACCF + b], 1);
      mbar_init(&bars[B_ACCE + b], 4);
    }
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = smem_u32(sm + OFF_A), b_base = smem_u32(sm + OFF_B);
  auto fail = [&]() {
    *abort_flag = 1;
    if (err != nullptr) atomicOr(err, ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t id = idesc_bf16(PT_M, PT_N, false, true);
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, WAIT_NS));
    };
    bool ok = true;
    int64_t g = 0;   // k-chunks issued (W stage counter)
    int seg = 0;     // token tiles started
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
      for (int kc = 0; kc < 8; ++kc, ++g) {
        const int st = (int)(g % NST);
        if (!wait(&bars[B_FULL + st], (uint32_t)((g / NST) & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // A: K-major chunk kc, 32 bytes per K = 16 step; B: MN-major, 64-column atoms
          // 8 KB apart, 8-row k groups 1 KB apart, 16 k-rows = 2 KB per step
          const uint64_t ad = smem_desc(a_base + kc * ACHUNK + kk * 32, 16, 1024, SW128);
          const uint64_t bd = smem_desc(b_base + st * STAGE + kk * 2048, 8192, 1024, SW128);
          mma_f16_warp(d, ad, bd, id, (kc | kk) != 0);
        }
        mma_commit_warp(&bars[B_EMPTY + st]);
      }
      if (!ok) break;
      mma_commit_warp(&bars[B_ACCF + buf]);
      const bool last = (f + 1 == f1) || ((f + 1) % NT == 0);
      if (last) mma_commit_warp(&bars[B_AFREE]);
    }
    if (!ok && lane == 0) fail();
    const int zero = 0;
    mma_commit_warp(&bars[B_DRAIN]);
    (void)mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- W producer
    bool ok = true;
    int64_t g = 0;
    for (int64_t f = f0; ok && f < f1; ++f) {
      const int x0 = (int)(f % NT) * PT_N;
      for (int kc = 0; kc < 8; ++kc, ++g) {
        const int st = (int)(g % NST);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_EMPTY + st],
                                               (uint32_t)((g / NST) & 1) ^ 1, abort_flag, WAIT_NS));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[B_FULL + st], STAGE);
          const uint32_t dst = b_base + st * STAGE;
#pragma unroll
          for (int a4 = 0; a4 < 4; ++a4)
            tma_load_2d(dst + a4 * 8192, &wmap, x0 + 64 * a4, 64 * kc, &bars[B_FULL + st]);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) fail();
    // let the requested loads land before the CTA can exit
    const int zero = 0;
    for (int64_t gg = (g > NST ? g - NST : 0); gg < g; ++gg)
      (void)mbar_wait(&bars[B_FULL + (int)(gg % NST)], (uint32_t)((gg / NST) & 1), &zero,
                      WAIT_NS);
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------- convert + epilogue
    const int q = warp & 3;                 // TMEM lane quarter
    const int row = q * 32 + lane;          // token row of the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int cw = warp - 4;
    const int rin = lane >> 2, sub = lane & 3;
    bool ok = true;
    int seg = 0;
    for (int64_t f = f0, u = 0; ok && f < f1; ++f, ++u) {
      const int64_t m = f / NT;
      const bool first = (f == f0) || (f % NT == 0);
      if (first) {
        // convert the token tile's codes (chunks cw and cw + 4) once
        if (seg > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_AFREE], (seg - 1) & 1, abort_flag, WAIT_NS));
          if (!ok) break;
        }
#pragma unroll 1
        for (int c = cw; c < 8; c += 4) {
          const uint32_t chunk = a_base + c * ACHUNK;
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int r = 8 * i + rin;
            const int64_t t = m * PT_M + r;
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (t < T) {
              const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
              if (slot >= 0 && slot < n_slots)
                x = __ldg(reinterpret_cast<const uint4*>(codes + slot * D + c * 64 + sub * 16));
              else if (err != nullptr && c == cw && i == 0)
                atomicOr(err, ERR_BLOCK_TABLE);  // a row with no slot reads as zeros
            }
            uint32_t h[8];
            h[0] = e4m3x2_to_bf16x2((uint16_t)(x.x & 0xFFFFu)); h[1] = e4m3x2_to_bf16x2((uint16_t)(x.x >> 16));
            h[2] = e4m3x2_to_bf16x2((uint16_t)(x.y & 0xFFFFu)); h[3] = e4m3x2_to_bf16x2((uint16_t)(x.y >> 16));
            h[4] = e4m3x2_to_bf16x2((uint16_t)(x.z & 0xFFFFu)); h[5] = e4m3x2_to_bf16x2((uint16_t)(x.z >> 16));
            h[6] = e4m3x2_to_bf16x2((uint16_t)(x.w & 0xFFFFu)); h[7] = e4m3x2_to_bf16x2((uint16_t)(x.w >> 16));
            const uint32_t o0 = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((2 * sub) ^ (r & 7)) << 4));
            const uint32_t o1 = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((2 * sub + 1) ^ (r & 7)) << 4));
            sts128p(chunk + o0, make_uint4(h[0], h[1], h[2], h[3]));
            sts128p(chunk + o1, make_uint4(h[4], h[5], h[6], h[7]));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_AREADY]);
        if (k_rope != nullptr && f % NT == 0) {
          // rows cw*32 .. cw*32+31 of the tile, four rows per pass, 8 codes per lane
          const int part = lane & 7;
#pragma unroll 1
          for (int i = 0; i < 8; ++i) {
            const int64_t t = m * PT_M + cw * 32 + 4 * i + (lane >> 3);
            if (t >= T) break;
            const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (slot >= 0 && slot < n_slots) {
              const uint2 x = __ldg(reinterpret_cast<const uint2*>(codes + slot * D + DL + part * 8));
              const float sR = __ldg(&scales[slot * 2 + 1]);
              e4m3x4_to_f32(x.x, v);
              e4m3x4_to_f32(x.y, v + 4);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[k] *= sR;
            }
            float4* dst = reinterpret_cast<float4*>(k_rope + t * DR + part * 8);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
        ++seg;
      }
      // epilogue of tile f: accumulator buffer u & 1
      const int buf = (int)(u & 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_ACCF + buf], (uint32_t)((u >> 1) & 1), abort_flag, WAIT_NS));
      if (!ok) break;
      tc_fence_after();
      const int64_t t = m * PT_M + row;
      float sL = 0.f;
      if (t < T) {
        const int64_t slot = slots != nullptr ? __ldg(&slots[t]) : t;
        if (slot >= 0 && slot < n_slots) sL = __ldg(&scales[slot * 2]);
      }
      uint16_t* yrow = y + t * (int64_t)N + (f % NT) * PT_N;
#pragma unroll 1
      for (int c = 0; c < PT_N; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + buf * PT_N + c, v);
        tmem_wait_ld();
        uint32_t p[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a0 = __uint_as_float(v[2 * j]) * sL, a1 = __uint_as_float(v[2 * j + 1]) * sL;
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p[j]) : "f"(a1), "f"(a0));
        }
        if (t < T) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + c);
          dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
          dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_ACCE + buf]);
    }
    if (!ok && lane == 0) fail();
  }
  // warps 2 and 3 have no role
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t make_w_map(const uint16_t* w, int N, CUtensorMap* map) {
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
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)PT_K};
  const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(w), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const uint8_t* codes, const float* scales, const int64_t* slots,
                           int64_t n_slots, int64_t T, const uint16_t* w, int N, uint16_t* y,
                           float* k_rope, unsigned* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap map;
  cudaError_t e = make_w_map(w, N, &map);
  if (e != cudaSuccess) return e;
  const int64_t tot = ((T + PT_M - 1) / PT_M) * (N / PT_N);
  const int grid = (int)(tot < NUM_SMS ? tot : NUM_SMS);
  prefill_kernel<<<grid, 256, SMEM, s>>>(codes, scales, slots, n_slots, T, N, y, k_rope, err, map);
  return cudaGetLastError();
}

}  // namespace kv8
