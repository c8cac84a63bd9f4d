// decode_tc.cu -- tcgen05 tensor-core split-T absorbed MLA decode over the e4m3
// latent cache, for one GB300 SM per CTA.
//
// Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description: the latent Lc is both key and value of the
// absorbed attention, the RoPE part Rc is key only, and each row's f32 scale is
// applied outside its dot product; closing note: split-T kernels for long caches.
// Per (sequence b, head h):
//   z_t = sm * ( sLc_t <q_lat, dec(Lc_t)> + sRc_t <q_rope, dec(Rc_t)> )
//   o   = sum_t softmax(z)_t sLc_t dec(Lc_t)
//
// One CTA = one work item (sequence, group of N heads, range of tiles); N in
// {16, 32, 64}.  Both contractions of a 128-token tile run on the tensor cores
// with f32 accumulators in TMEM; the per-row scales stay outside the MMA:
//   S^T[t][h] = K_t . Q_h      kind::f16, M = 128 tokens, N heads, K = 512 (S_L)
//                              and 64 (S_R); K converted from e4m3 to fp16 (exact),
//                              Q in fp16 with a per-head power-of-two scale
//   z[t][h]   = c_h (sLc_t S_L + sRc_t S_R)                  (softmax warps)
//   P''[h][t] = 2^(z - m_h) (sLc_t / s_ref) P_TOP            (two e4m3 terms hi + lo)
//   O^T[d][h] += sum_t V[t][d] P''[h][t]   kind::f8f6f4, M = 128 latent rows (x4),
//                              N heads, K = 128 tokens; V^T is the e4m3 cache tile
//                              itself (MN-major), loaded by TMA, never converted
// The fp16 score operand: one chunk of 128 tokens x 64 channels (128-byte
// swizzle, K-major).  The e4m3 context operand: one d-block of 128 tokens x 128
// channels (the TMA box, 128-byte swizzle), read as V^T.
//
// Warp roles (14 warps; 16 for 16-head groups, which have six converters):
//   warp 0       issues the score MMAs of every tile (lane 0 alone, or for N = 16
//                the whole warp with one elected lane); the warp owns TMEM.
//   last warp    loads each tile's four e4m3 d-blocks by TMA (the next tile's
//                block as soon as this tile's MMAs on it are done), zeroes rows
//                that hold no data, and issues the context MMAs as soon as the
//                tile's P'' is written.
//   warps 1-8    softmax, two groups of four warps; a thread owns one token row
//                (its TMEM lane) and half of the heads: tile max per head by a
//                transposed warp reduction, running denominators per thread, lazy
//                rescaling of O (only the heads whose max grew by more than 2^1, or
//                whose tile max lies more than 2^10 below it),
//                P'' split into e4m3 hi + lo in f16 arithmetic.
//   warps 9..     score converters: the chunks Lc 0..7, Rc of every tile, in order,
//                into a 4-slot (6 for 16 heads) fp16 ring, one warp per slot (16-byte
//                loads, the next chunk's loads in flight while it waits for its
//                slot, hardware cvt, swizzled 16-byte stores).  The bulk-copy
//                engine prefetches tiles into L2 three tiles ahead.
// The ring has one consumer taking its chunks in order, so the parity waits on
// a slot are exact.  The scores of tile i+1 run on the tensor cores while the
// softmax of tile i runs on the CUDA cores.  Every wait is bounded (2 s): on a
// timeout the CTA flags the workspace error word, drains its MMAs and its TMA
// loads, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

using namespace ptx;

constexpr int CHUNK = TILE * 64 * 2;         // 16 KB: 128 rows x 64 fp16
constexpr int VBLK = TILE * 128;             // 16 KB: 128 rows x 128 e4m3 (one d-block of V)
constexpr int S_PER_TILE = 9;                // Lc channel blocks 0..7, then Rc
constexpr int NSOFT = 8;
constexpr int WARP_SOFT = 1;
constexpr int WARP_CONV = WARP_SOFT + NSOFT;  // first converter warp (9)
constexpr int NBAR_ALLOC = 48;               // mbarriers allocated

// Per head-group width: the score ring and its converter warps (one warp per
// slot).  16-head groups leave room in shared memory for six slots, half as many
// e4m3 bytes again in flight; six converters keep the block at 16 warps, four per
// SM sub-partition, so each thread keeps 128 registers (eight slots and 18 warps
// would cap them at 96 and spill).
template <int N>
struct Cfg {
  static constexpr int S_RING = (N <= 16) ? 6 : 4;        // score-operand chunk slots
  static constexpr int NCONV = S_RING;
  static constexpr int WARP_VMMA = WARP_CONV + NCONV;     // V tile loads and context MMAs
  static constexpr int NTHREADS = (WARP_VMMA + 1) * 32;
  // barrier indices
  static constexpr int B_SF = 0;                      // [S_RING] score chunk converted
  static constexpr int B_SE = B_SF + S_RING;          // [S_RING] score chunk consumed
  static constexpr int B_VT = B_SE + S_RING;          // [4] e4m3 d-block loaded (TMA transactions)
  static constexpr int B_VD = B_VT + 4;               // [4] context MMAs on a d-block done
  static constexpr int B_S_FULL = B_VD + 4;           // [2] scores of a tile in TMEM
  static constexpr int B_S_EMPTY = B_S_FULL + 2;      // [2] scores read by the softmax
  static constexpr int B_P_FULL = B_S_EMPTY + 2;      // P'' of a tile written
  static constexpr int B_O_DONE = B_P_FULL + 1;       // context MMAs of a tile done
  static constexpr int B_G = B_O_DONE + 1;            // [group][2] softmax group barriers
  static constexpr int B_DRAIN = B_G + 4;             // [2] issuers' final drains
  static_assert(B_DRAIN + 2 <= NBAR_ALLOC, "barrier layout exceeds the barriers allocated");
};
constexpr int L2_AHEAD = 3;                  // tiles prefetched into L2 ahead of the converters
// Lazy rescaling thresholds.  The e4m3 weights P'' = 2^(z - m) (sLc / s_ref)
// P_TOP are at most 2^TAU * TAU_S_POW * P_TOP = 256 <= 448, and with this
// little headroom the largest weights of a tile sit near the top of the e4m3
// range, where the two-term split keeps about 8 significant bits.
constexpr float TAU = 1.0f;                  // rescale O if a head's max grows by > 2^1
constexpr float TAU_S_POW = 2.0f;            // ... or the scale reference by > 2
constexpr float P_TOP = 64.0f;
// A head's running max also moves down, to a tile's max that lies more than
// 2^DOWN below it (and within 2^DOWN_CAP of the highest max so far): the weights
// of a bulk of tokens far below an earlier dominant token then stay inside the
// e4m3 range instead of flushing to zero in both terms.
constexpr float DOWN = 10.0f;
constexpr float DOWN_CAP = 60.0f;
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on any single wait
constexpr float LOG2E = 1.4426950408889634f;

constexpr int align1k(int x) { return (x + 1023) & ~1023; }

template <int N>
struct Lay {
  static constexpr int NH = N / 2;                         // heads per softmax group
  static constexpr int Q = 0;                              // 9 chunks [N x 64] fp16
  static constexpr int RINGO = align1k(Q + 9 * N * 128);
  static constexpr int VT = RINGO + Cfg<N>::S_RING * CHUNK; // e4m3 V tile: 4 d-blocks
  static constexpr int P = VT + 4 * VBLK;                   // e4m3 P'' hi, lo: [N x 128 tokens] each
  static constexpr int BAR = P + 2 * N * 128;              // NBAR_ALLOC mbarriers
  static constexpr int FLAGS = BAR + NBAR_ALLOC * 8;       // tmem base, abort, corr flags
  static constexpr int CS = FLAGS + 32;                    // score constant per head
  static constexpr int MU = CS + N * 4;                    // max in use per head (log2)
  static constexpr int MHI = MU + N * 4;                   // highest max in use so far per head
  static constexpr int ALPHA = MHI + N * 4;                // rescale of l this tile
  static constexpr int FCOL = ALPHA + N * 4;               // rescale of O columns this tile
  static constexpr int LFIN = FCOL + N * 4;                // final denominators
  static constexpr int RMAX = LFIN + N * 4;                // [4][N] per-warp tile maxima
  static constexpr int RS = RMAX + 4 * N * 4;              // [2][4] warp max of sLc
  static constexpr int TOTAL = RS + 32;
  static constexpr int TMEM_COLS = (8 * N <= 128) ? 128 : (8 * N <= 256 ? 256 : 512);
};



__device__ __forceinline__ uint4 ldg16(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void sts8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Offset of 16-byte unit u of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

// Transposed warp reduction of NV <= 32 values per lane: afterwards lane holds
// the reduction over the 32 lanes of value index (lane >> (5 - log2 NV)).
template <int NV, bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(const float (&v)[NV], int lane) {
  static_assert(NV >= 2 && NV <= 32 && (NV & (NV - 1)) == 0, "NV must be a power of two");
  float t[NV / 2];
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int j = 0; j < NV / 2; ++j) {
      const float send = up ? v[j] : v[j + NV / 2];
      const float keep = up ? v[j + NV / 2] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      t[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  int n = NV / 2;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < NV / 4; ++j) {
        if (j < n / 2) {
          const float send = up ? t[j] : t[j + n / 2];
          const float keep = up ? t[j + n / 2] : t[j];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          t[j] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
      }
      n >>= 1;
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, t[0], o);
      t[0] = MAX ? fmaxf(t[0], recv) : t[0] + recv;
    }
  }
  return t[0];
}

template <int N>
__global__ void __launch_bounds__(Cfg<N>::NTHREADS, 1)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
  using L = Lay<N>;
  using C = Cfg<N>;
  constexpr int S_RING = C::S_RING, NCONV = C::NCONV, WARP_VMMA = C::WARP_VMMA,
                NTHREADS = C::NTHREADS;
  constexpr int B_SF = C::B_SF, B_SE = C::B_SE, B_VT = C::B_VT, B_VD = C::B_VD,
                B_S_FULL = C::B_S_FULL, B_S_EMPTY = C::B_S_EMPTY, B_P_FULL = C::B_P_FULL,
                B_O_DONE = C::B_O_DONE, B_G = C::B_G, B_DRAIN = C::B_DRAIN;
  constexpr int NH = L::NH;
  constexpr int LOG2_NH = NH == 8 ? 3 : (NH == 16 ? 4 : 5);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ WorkItem s_it;
  __shared__ int s_ok;
  if (warp == 0) {
    WorkItem it;
    const bool ok = find_item(a, blockIdx.x, it);
    if (lane == 0 && ok) record_segment(a, blockIdx.x, it);
    if (lane == 0) {
      s_it = it;
      s_ok = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;  // past the last work item of this call
  const int g_head = s_it.g, b = s_it.b;
  const int64_t t0 = s_it.t0, t_end = s_it.t1;
  const int n_tiles = (int)((t_end - t0 + TILE - 1) / TILE);
  const int h0 = g_head * N;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::FLAGS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::FLAGS + 4);
  volatile int* corr_flag = reinterpret_cast<volatile int*>(sm + L::FLAGS + 8);  // [2][2]
  float* cs = reinterpret_cast<float*>(sm + L::CS);
  float* mu_s = reinterpret_cast<float*>(sm + L::MU);
  float* alpha_s = reinterpret_cast<float*>(sm + L::ALPHA);
  float* fcol = reinterpret_cast<float*>(sm + L::FCOL);
  float* lfin = reinterpret_cast<float*>(sm + L::LFIN);
  float* rmax = reinterpret_cast<float*>(sm + L::RMAX);
  float* rs = reinterpret_cast<float*>(sm + L::RS);

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < S_RING; ++i) {
      mbar_init(&bars[B_SF + i], 1);
      mbar_init(&bars[B_SE + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[B_VT + i], 1);
      mbar_init(&bars[B_VD + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], NSOFT);
    }
    mbar_init(&bars[B_P_FULL], NSOFT);
    mbar_init(&bars[B_O_DONE], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_G + i], NSOFT / 2);
    mbar_init(&bars[B_DRAIN], 1);
    mbar_init(&bars[B_DRAIN + 1], 1);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) corr_flag[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < N) {
    mu_s[threadIdx.x] = -INFINITY;
    reinterpret_cast<float*>(sm + L::MHI)[threadIdx.x] = -INFINITY;
  }
  // Query -> fp16, one warp per head, with a per-head power-of-two scale that
  // puts max|q| in [2^14, 2^15); c_h undoes it and folds in sm_scale*log2(e).
  if (warp >= 1) {
    const uint32_t qbase = smem_u32(sm + L::Q);
    for (int hh = warp - 1; hh < N; hh += (NTHREADS / 32) - 1) {
      const int h = h0 + hh;
      float v[16], r[2];
      if (h < a.H) {
        const float4* ql =
            reinterpret_cast<const float4*>(a.q_lat + ((int64_t)b * a.H + h) * DL) + lane * 4;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 x = __ldg(ql + k);
          v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
        }
        const float2 y = __ldg(reinterpret_cast<const float2*>(
            a.q_rope + ((int64_t)b * a.H + h) * DR + 2 * lane));
        r[0] = y.x; r[1] = y.y;
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0.f;
        r[0] = r[1] = 0.f;
      }
      float amax = fmaxf(fabsf(r[0]), fabsf(r[1]));
#pragma unroll
      for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int e = 0;
      if (amax > 0.f && isfinite(amax)) {
        int x;
        frexpf(amax, &x);
        e = min(max(15 - x, -120), 120);
      }
      const float sc = ldexpf(1.0f, e);
      uint32_t hv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __half2 hh2 = __floats2half2_rn(v[2 * k] * sc, v[2 * k + 1] * sc);
        hv[k] = *reinterpret_cast<const uint32_t*>(&hh2);
      }
      const int c = lane >> 2, u = 2 * (lane & 3);
      const uint32_t rowbase = qbase + c * N * 128;
      sts128(rowbase + sw128(hh, u), make_uint4(hv[0], hv[1], hv[2], hv[3]));
      sts128(rowbase + sw128(hh, u + 1), make_uint4(hv[4], hv[5], hv[6], hv[7]));
      const __half2 rr = __floats2half2_rn(r[0] * sc, r[1] * sc);
      const uint32_t ra = qbase + 8 * N * 128 + sw128(hh, lane >> 2) + (lane & 3) * 4;
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(ra), "r"(*reinterpret_cast<const uint32_t*>(&rr))
                   : "memory");
      if (lane == 0) cs[hh] = (h < a.H) ? a.sm_scale * LOG2E / sc : 0.f;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sring = smem_u32(sm + L::RINGO);
  const uint32_t vtile = smem_u32(sm + L::VT);
  const uint32_t p_base = smem_u32(sm + L::P);
  const uint32_t q_base = smem_u32(sm + L::Q);

  if (warp == 0) {
    // ---------------------------------------------------------- score MMAs
    // Narrow head groups (light softmax) issue from the whole converged warp with
    // elect.sync; wider ones from lane 0 alone, which leaves more issue slots to
    // the softmax warps that share the SM sub-partition (measured both ways on
    // the workloads of each width).
    constexpr bool WARP_ISSUE = (N <= 16);
    if (WARP_ISSUE || lane == 0) {
      const uint32_t idS = idesc_f16(128, N, false, false);
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait(bar, parity, abort_flag, WAIT_NS);
        if constexpr (WARP_ISSUE) return __all_sync(0xffffffffu, ok);
        return ok;
      };
      auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
        if constexpr (WARP_ISSUE) mma_f16_warp(d, ad, bd, id, acc);
        else mma_f16(d, ad, bd, id, acc);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (WARP_ISSUE) mma_commit_warp(bar);
        else mma_commit(bar);
      };
      // The ring has this one consumer taking its chunks in order, so a parity
      // wait on a slot is never more than one phase ahead of the slot.  Within a
      // tile the loop runs straight through; a failed wait only marks the tile
      // bad (the abort flag then makes every later wait return at once).
      bool ok = true;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int buf = i & 1;
        if (!wait(&bars[B_S_EMPTY + buf], ((i >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dL = tmem + buf * 2 * N, dR = dL + N;
        for (int c = 0; c < S_PER_TILE; ++c) {
          const int sc = i * S_PER_TILE + c, slot = sc % S_RING;
          ok = wait(&bars[B_SF + slot], (sc / S_RING) & 1) && ok;
          tc_fence_after();
          const uint32_t ab = sring + slot * CHUNK, bb = q_base + c * N * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma(c < 8 ? dL : dR, smem_desc(ab + kk * 32, 16, 1024, SW128),
                smem_desc(bb + kk * 32, 16, 1024, SW128), idS, (c == 8 ? kk : (c | kk)) != 0);
          commit(&bars[B_SE + slot]);
        }
        if (ok) commit(&bars[B_S_FULL + buf]);
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        atomicOr(a.err, ERR_TIMEOUT);
      }
      // drain: every MMA issued above completes before TMEM is released (this
      // wait ignores the abort flag; it is still bounded in time)
      const int zero = 0;
      commit(&bars[B_DRAIN]);
      (void)mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
    }
    __syncwarp();
  } else if (warp == WARP_VMMA) {
    // ---------------------------------------------------------- context MMAs
    // The e4m3 Lc bytes of a tile come straight from the cache by TMA (128-byte
    // swizzle), one [128 tokens x 128 channels] d-block per barrier; rows past
    // the data are zeroed here.  O^T[d][h] += V^T P''^T with A = V^T (MN-major
    // e4m3) and B = P'' in two e4m3 terms (hi + lo), K = 32 tokens per MMA.  The
    // next tile's d-block m is requested as soon as this tile's MMAs on it are
    // done.  The whole warp walks the loop; one elected lane issues.
    const uint32_t idV = idesc_f16(128, N, true, false);  // e4m3 encodes as format 0
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, WAIT_NS));
    };
    int64_t s0 = -1, s1 = -1;
    int nv = 0;
    auto tile_rows = [&](int i) {
      const int64_t tb = t0 + (int64_t)i * TILE;
      const int64_t n = t_end - tb;
      nv = n < TILE ? (int)n : TILE;
      s0 = slot_of(a, b, tb);
      s1 = nv > PAGE ? slot_of(a, b, tb + PAGE) : -1;
    };
    auto load_block = [&](int m) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[B_VT + m], (s0 >= 0 ? 8192u : 0u) + (s1 >= 0 ? 8192u : 0u));
        const uint32_t dst = vtile + m * VBLK;
        if (s0 >= 0) tma_load_2d(dst, &tmap, 128 * m, (int)s0, &bars[B_VT + m]);
        if (s1 >= 0) tma_load_2d(dst + 8192, &tmap, 128 * m, (int)s1, &bars[B_VT + m]);
      }
      __syncwarp();
    };
    auto zero_rows = [&](int m, int r0, int r1) {  // rows [r0, r1) of d-block m
      const uint32_t base = vtile + m * VBLK;
      for (int u = r0 * 8 + lane; u < r1 * 8; u += 32) sts128(base + u * 16, make_uint4(0u, 0u, 0u, 0u));
    };
    bool ok = true;
    int requested = 1;  // tiles whose four d-blocks have been requested
    tile_rows(0);
    for (int m = 0; m < 4; ++m) load_block(m);
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (!wait(&bars[B_P_FULL], i & 1)) { ok = false; break; }
      tc_fence_after();
      for (int m = 0; m < 4; ++m) {
        ok = wait(&bars[B_VT + m], i & 1) && ok;
        if (s0 < 0 || s1 < 0 || nv < TILE) {
          // rows with no data (past the end, or a page the block table does not map)
          if (s0 < 0) zero_rows(m, 0, nv < PAGE ? nv : PAGE);
          if (s1 < 0 && nv > PAGE) zero_rows(m, PAGE, nv);
          if (nv < TILE) zero_rows(m, nv, TILE);
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        const uint32_t vb = vtile + m * VBLK;
        const uint32_t d = tmem + 4 * N + m * N;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // A = V^T: 128 channels (one swizzle atom) x 32 tokens, 8-token groups 1 KB apart
          const uint64_t ad = smem_desc(vb + kk * 4096, VBLK, 1024, SW128);
#pragma unroll
          for (int term = 0; term < 2; ++term) {
            const uint64_t bd = smem_desc(p_base + term * N * 128 + kk * 32, 16, 1024, SW128);
            mma_f8_warp(d, ad, bd, idV, (i > 0 || kk > 0 || term > 0) ? 1u : 0u);
          }
        }
        mma_commit_warp(&bars[B_VD + m]);
      }
      if (!ok) break;
      mma_commit_warp(&bars[B_O_DONE]);
      if (i + 1 < n_tiles) {
        tile_rows(i + 1);
        for (int m = 0; m < 4; ++m) {
          ok = wait(&bars[B_VD + m], i & 1) && ok;
          load_block(m);
        }
        ++requested;
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    }
    const int zero = 0;
    mma_commit_warp(&bars[B_DRAIN + 1]);
    (void)mbar_wait(&bars[B_DRAIN + 1], 0, &zero, WAIT_NS);
    // after an abort the last tile's loads may still be in flight: let them land
    // (a completed phase passes at once; this wait ignores the abort flag)
    if (!ok) {
      for (int m = 0; m < 4; ++m)
        (void)mbar_wait(&bars[B_VT + m], (requested - 1) & 1, &zero, WAIT_NS);
    }
    __syncwarp();
  } else if (warp < WARP_CONV) {
    // ---------------------------------------------------------- softmax
    const int grp = (warp - WARP_SOFT) >> 2;      // head group: heads [grp*NH, grp*NH + NH)
    const int wq = (warp - WARP_SOFT) & 3;        // warp within the group
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;          // token row of the tile = TMEM lane
    const int st = wq * 32 + lane;                // thread within the group
    const int hb = grp * NH;                      // first head of the group
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    float lpart[NH];  // running softmax denominators of this thread's token rows
#pragma unroll
    for (int h = 0; h < NH; ++h) lpart[h] = 0.f;
    float sref = 0.f;
    bool ok = true;
    // group barriers k = 0, 1: each counts its own phases
    int gph[2] = {0, 0};
    auto group_sync = [&](int k) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_G + 2 * grp + k]);
      return mbar_wait_warp(&bars[B_G + 2 * grp + k], (gph[k]++) & 1, abort_flag, WAIT_NS);
    };
    // byte of P''[h][t] (K-major [N x 128 tokens], 128-byte swizzle): row h,
    // 16-byte unit t >> 4, byte t & 15; the lo term follows the hi term
    auto p_addr = [&](int h) -> uint32_t {
      return p_base + (uint32_t)((h >> 3) * 1024 + (h & 7) * 128 + (((row >> 4) ^ (h & 7)) << 4) +
                                 (row & 15));
    };
    const float4* cs4 = reinterpret_cast<const float4*>(cs + hb);
    const float4* mu4 = reinterpret_cast<const float4*>(mu_s + hb);
    const float4* al4 = reinterpret_cast<const float4*>(alpha_s + hb);
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int64_t tok = t0 + (int64_t)i * TILE + row;
      float sL = 0.f, sR = 0.f;
      bool valid = false;
      if (tok < t_end) {
        const int64_t slot = slot_of(a, b, tok);
        if (slot >= 0) {
          const float2 s2 = __ldg(reinterpret_cast<const float2*>(a.scales + slot * 2));
          sL = s2.x;
          sR = s2.y;
          valid = true;
        }
      }
      const int buf = i & 1;
      if (!mbar_wait_warp(&bars[B_S_FULL + buf], (i >> 1) & 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // u = sLc S_L + sRc S_R; the score in log2 units is z = c_h u with c_h >= 0,
      // so the tile max is taken on u and c_h is applied inside the exponent
      float z[NH];
#pragma unroll
      for (int c = 0; c < NH; c += 8) {
        uint32_t rl[8], rr[8];
        tmem_ld8(tmem + lane_addr + buf * 2 * N + hb + c, rl);
        tmem_ld8(tmem + lane_addr + buf * 2 * N + N + hb + c, rr);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          z[c + j] = valid ? fmaf(sR, __uint_as_float(rr[j]), sL * __uint_as_float(rl[j]))
                           : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_EMPTY + buf]);

      // Tile max per head (and of sLc) over the group's four warps.  The running
      // max of a head moves (and its O columns are rescaled) only if the tile max
      // exceeds it by more than 2^TAU, the scale reference only if a scale
      // exceeds it TAU_S_POW times.
      bool corr = false;
      {
        const float mx = warp_transpose_reduce<NH, true>(z, lane);
        if ((lane & ((32 >> LOG2_NH) - 1)) == 0)
          rmax[wq * N + hb + (lane >> (5 - LOG2_NH))] = mx;
        float smax = valid ? sL : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) rs[grp * 4 + wq] = smax;
        if (st == 0) corr_flag[grp * 2 + buf] = 0;
        if (!group_sync(0)) { ok = false; break; }
        const float gmax = fmaxf(fmaxf(rs[grp * 4 + 0], rs[grp * 4 + 1]),
                                 fmaxf(rs[grp * 4 + 2], rs[grp * 4 + 3]));
        const float sref_new = (gmax > sref * TAU_S_POW) ? gmax : sref;
        const float beta = (sref_new == sref) ? 1.f : (sref > 0.f ? sref / sref_new : 0.f);
        if (st < NH) {
          const int hh = hb + st;
          const float umax =
              fmaxf(fmaxf(rmax[hh], rmax[N + hh]), fmaxf(rmax[2 * N + hh], rmax[3 * N + hh]));
          const float tmax = (cs[hh] > 0.f) ? cs[hh] * umax : -INFINITY;
          float mu = mu_s[hh];
          float* mhi = reinterpret_cast<float*>(sm + L::MHI) + hh;
          float mn = mu;
          if (tmax > mu + TAU) {
            mn = tmax;
          } else if (tmax < mu - DOWN && tmax >= *mhi - DOWN_CAP && tmax > -INFINITY) {
            mn = tmax;
          }
          float alpha = 1.f;
          if (mn != mu) {
            alpha = (mu == -INFINITY) ? 0.f : ex2_approx(mu - mn);
            mu = mn;
          }
          *mhi = fmaxf(*mhi, mu);
          mu_s[hh] = mu;
          alpha_s[hh] = alpha;
          fcol[hh] = alpha * beta;
          if (i > 0 && alpha * beta != 1.f) corr_flag[grp * 2 + buf] = 1;
        }
        sref = sref_new;
        if (!group_sync(1)) { ok = false; break; }
        corr = corr_flag[grp * 2 + buf] != 0;
      }

      // probabilities; running denominators; P'' = p * (sLc / s_ref) * P_TOP
      // (a running max still at -inf is floored so that an empty row gives 2^-inf = 0)
      const float w = valid ? sL * (sref > 0.f ? P_TOP / sref : 0.f) : 0.f;
#pragma unroll
      for (int h = 0; h < NH; h += 4) {
        const float4 m4 = mu4[h / 4];
        const float4 a4 = al4[h / 4];
        const float4 c4 = cs4[h / 4];
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w}, aa[4] = {a4.x, a4.y, a4.z, a4.w};
        const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = ex2_approx(fmaf(cc[j], z[h + j], -fmaxf(mm[j], -3.0e38f)));
          lpart[h + j] = fmaf(lpart[h + j], aa[j], p);
          z[h + j] = p * w;
        }
      }
      // e4m3 weights P'' as hi + lo on the same scale, computed in
      // f16 (the residual of the hi term is exact there); bytes packed by head
      uint32_t phi[NH / 4], plo[NH / 4];
#pragma unroll
      for (int h = 0; h < NH; h += 4) {
        const __half2 x01 = __floats2half2_rn(z[h], z[h + 1]);
        const __half2 x23 = __floats2half2_rn(z[h + 2], z[h + 3]);
        const uint16_t h01 = f16x2_to_e4m3x2(x01), h23 = f16x2_to_e4m3x2(x23);
        const uint32_t d01 = e4m3x2_to_f16x2(h01), d23 = e4m3x2_to_f16x2(h23);
        const uint16_t l01 = f16x2_to_e4m3x2(__hsub2(x01, *reinterpret_cast<const __half2*>(&d01)));
        const uint16_t l23 = f16x2_to_e4m3x2(__hsub2(x23, *reinterpret_cast<const __half2*>(&d23)));
        phi[h / 4] = (uint32_t)h01 | ((uint32_t)h23 << 16);
        plo[h / 4] = (uint32_t)l01 | ((uint32_t)l23 << 16);
      }
      if (i > 0) {
        if (!mbar_wait_warp(&bars[B_O_DONE], (i - 1) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (corr) {
          // rescale the O columns of the heads whose factor moved, 8 heads at a
          // time, the four d-blocks' loads in flight together
#pragma unroll 1
          for (int c = 0; c < NH; c += 8) {
            const float4 f0 = *reinterpret_cast<const float4*>(fcol + hb + c);
            const float4 f1 = *reinterpret_cast<const float4*>(fcol + hb + c + 4);
            const float ff[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
            bool moved = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) moved |= (ff[j] != 1.f);
            if (!moved) continue;  // the same for every thread of the group
            uint32_t r[4][8];
#pragma unroll
            for (int m = 0; m < 4; ++m) tmem_ld8(tmem + lane_addr + 4 * N + m * N + hb + c, r[m]);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int j = 0; j < 8; ++j) r[m][j] = __float_as_uint(__uint_as_float(r[m][j]) * ff[j]);
              tmem_st8(tmem + lane_addr + 4 * N + m * N + hb + c, r[m]);
            }
          }
          tmem_wait_st();
        }
      }
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const uint32_t ad = p_addr(hb + h);
        sts8(ad, phi[h / 4] >> (8 * (h & 3)));
        sts8(ad + N * 128, plo[h / 4] >> (8 * (h & 3)));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P_FULL]);
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    } else if (mbar_wait_warp(&bars[B_O_DONE], (n_tiles - 1) & 1, abort_flag, WAIT_NS)) {
      // denominators: reduce the per-thread partials of each head over the 128 rows
      {
        const float ls = warp_transpose_reduce<NH, false>(lpart, lane);
        if ((lane & ((32 >> LOG2_NH) - 1)) == 0)
          rmax[wq * N + hb + (lane >> (5 - LOG2_NH))] = ls;
      }
      if (group_sync(0)) {
        if (st < NH) {
          const int hh = hb + st;
          lfin[hh] = (rmax[hh] + rmax[N + hh]) + (rmax[2 * N + hh] + rmax[3 * N + hh]);
        }
        if (group_sync(1)) {
          // epilogue: unnormalised partial o = acc * s_ref / P_TOP, with (m, l) per head
          const float oscale = sref * (1.0f / P_TOP);
          tc_fence_after();
          const int64_t base = (int64_t)blockIdx.x * N;  // this item's partials
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int c = 0; c < NH; c += 8) {
              uint32_t r[8];
              tmem_ld8(tmem + lane_addr + 4 * N + m * N + hb + c, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int h = hb + c + j;
                if (h0 + h < a.H)
                  a.ws_o[(base + h) * DL + m * 128 + row] = __uint_as_float(r[j]) * oscale;
              }
            }
          }
          if (st < NH && h0 + hb + st < a.H) {
            a.ws_m[base + hb + st] = mu_s[hb + st];
            a.ws_l[base + hb + st] = lfin[hb + st];
          }
        } else {
          ok = false;
        }
      } else {
        ok = false;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, ERR_TIMEOUT);
      }
    } else {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    }
  } else {
    // ---------------------------------------------------------- converters
    // The converters fill the score ring with the fp16 chunks of every tile in
    // order (Lc blocks 0..7, then Rc); converter w takes every NCONV-th chunk.
    // Lane l handles rows 8i + (l >> 2) (i = 0..15) and 16-byte piece (l & 3) of
    // the chunk's 64 bytes per row; rows 0..63 are the tile's first page,
    // 64..127 its second.
    constexpr bool score_side = true;
    const int cw = warp - WARP_CONV;
    constexpr int nconv = NCONV;
    constexpr int per_tile = S_PER_TILE;
    constexpr int ring = S_RING;
    const uint32_t ring_base = sring;
    uint64_t* full = &bars[B_SF];
    uint64_t* empty = &bars[B_SE];
    const int total = per_tile * n_tiles;
    const int rin = lane >> 2, sub = lane & 3;
    int ctile[2] = {-1, -1};
    const uint8_t* cpg[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
    int cvalid[2] = {0, 0};
    // page base pointers (or null) and valid row count of a tile, with a 2-entry cache
    auto pages_of = [&](int tile, const uint8_t*& p0, const uint8_t*& p1, int& nvalid) {
      if (ctile[0] == tile) { p0 = cpg[0][0]; p1 = cpg[0][1]; nvalid = cvalid[0]; return; }
      if (ctile[1] == tile) { p0 = cpg[1][0]; p1 = cpg[1][1]; nvalid = cvalid[1]; return; }
      const int64_t tb = t0 + (int64_t)tile * TILE;
      const int64_t nv = (t_end - tb < TILE) ? t_end - tb : TILE;
      const uint8_t* q[2];
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        q[pg] = nullptr;
        if (pg * PAGE < nv) {
          const int64_t slot = slot_of(a, b, tb + pg * PAGE);
          if (slot >= 0) q[pg] = a.codes + slot * D;
        }
      }
      ctile[1] = ctile[0]; cpg[1][0] = cpg[0][0]; cpg[1][1] = cpg[0][1]; cvalid[1] = cvalid[0];
      ctile[0] = tile; cpg[0][0] = q[0]; cpg[0][1] = q[1]; cvalid[0] = (int)nv;
      p0 = q[0]; p1 = q[1]; nvalid = (int)nv;
    };
    auto prefetch_tile = [&](int tile) {
      const int64_t tb = t0 + (int64_t)tile * TILE;
      for (int pg = 0; pg < 2; ++pg) {
        const int64_t tk = tb + pg * PAGE;
        if (tk >= t_end) break;
        const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
        const int64_t slot = slot_of(a, b, tk);
        if (slot >= 0) prefetch_l2(a.codes + slot * D, (uint32_t)(nt * D));
      }
    };
    uint4 dat[16];
    auto load = [&](int j) {
      const int tile = j / per_tile, c = j % per_tile;
      const uint8_t *p0, *p1;
      int nv;
      pages_of(tile, p0, p1, nv);
      const int off = c * 64 + sub * 16;  // c == 8 is the Rc block: channels 512..575
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 8 * i + rin;
        const uint8_t* pg = (i < 8) ? p0 : p1;
        dat[i] = (pg != nullptr && r < nv) ? ldg16(pg + (size_t)(r & 63) * D + off)
                                           : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    bool ok = true;
    if (score_side && cw == 0 && lane == 0) {
      // the first tiles' lines: ask the bulk-copy engine for them up front
      for (int tl = 0; tl < L2_AHEAD && tl < n_tiles; ++tl) prefetch_tile(tl);
    }
    if (cw < total) load(cw);
    for (int j = cw; j < total && ok; j += nconv) {
      const int slot = j % ring;
      const uint32_t slot_addr = ring_base + slot * CHUNK;
      if (!mbar_wait_warp(&empty[slot], ((j / ring) & 1) ^ 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 8 * i + rin;
        const uint4 x = dat[i];
        uint32_t h[8];
        h[0] = e4m3x2_to_f16x2((uint16_t)(x.x & 0xFFFFu)); h[1] = e4m3x2_to_f16x2((uint16_t)(x.x >> 16));
        h[2] = e4m3x2_to_f16x2((uint16_t)(x.y & 0xFFFFu)); h[3] = e4m3x2_to_f16x2((uint16_t)(x.y >> 16));
        h[4] = e4m3x2_to_f16x2((uint16_t)(x.z & 0xFFFFu)); h[5] = e4m3x2_to_f16x2((uint16_t)(x.z >> 16));
        h[6] = e4m3x2_to_f16x2((uint16_t)(x.w & 0xFFFFu)); h[7] = e4m3x2_to_f16x2((uint16_t)(x.w >> 16));
        sts128(slot_addr + sw128(r, 2 * sub), make_uint4(h[0], h[1], h[2], h[3]));
        sts128(slot_addr + sw128(r, 2 * sub + 1), make_uint4(h[4], h[5], h[6], h[7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[slot]);
      if (j + nconv < total) load(j + nconv);
      // L2 prefetch of the tile L2_AHEAD tiles ahead, when its score chunk 0 is converted
      const int tile = j / per_tile;
      if (score_side && lane == 0 && j % per_tile == 0 && tile + L2_AHEAD < n_tiles)
        prefetch_tile(tile + L2_AHEAD);
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

template <int N>
cudaError_t launch_n(const DecodeArgs& a, cudaStream_t s) {
  const int smem = Lay<N>::TOTAL + 1024;
  static std::atomic<int> memo[MAX_DEVICES];
  int done = 0;
  cudaError_t e = per_device(memo, [smem](int* v) {
    *v = 1;
    return cudaFuncSetAttribute(decode_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
  }, &done);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  e = make_cache_map(a, &map);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<N><<<a.plan.max_items, Cfg<N>::NTHREADS, smem, s>>>(a, map);
  return cudaGetLastError();
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to
// libcuda), then the map: `rank` dimensions, row strides in bytes (rank - 1 of
// them), unit element strides, rows past the extent read as zeros.
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, unsigned rank, void* base,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                         CUtensorMapSwizzle swizzle) {
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
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, type, rank, base, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of the e4m3 cache for the tile loads: rows of 576 bytes, boxes of
// 64 rows (one page) x 128 bytes (one channel block), 128-byte swizzle.  Rows
// (and columns) past the end of the map read as zeros.
cudaError_t make_cache_map(const DecodeArgs& a, CUtensorMap* map) {
  const int64_t rows = a.block_table != nullptr ? a.n_blocks * PAGE : a.T_contig;
  if (rows < 1 || a.codes == nullptr) {
    // no cache rows: no tile is ever loaded, the map is never read
    memset(map, 0, sizeof(*map));
    return cudaSuccess;
  }
  if (rows >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D};
  const cuuint32_t box[2] = {128, PAGE};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.codes), dims,
                      strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tc_available() { return true; }

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  switch (a.plan.hg) {
    case 16: return launch_n<16>(a, s);
    case 32: return launch_n<32>(a, s);
    case 64: return launch_n<64>(a, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kv8
