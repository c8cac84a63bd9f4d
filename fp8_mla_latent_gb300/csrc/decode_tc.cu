// decode_tc.cu -- tcgen05 tensor-core split-T absorbed MLA decode over the e4m3
// latent cache, for one GB300 SM per CTA.
//
// Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description: the latent Lc is both key and value of the
// absorbed attention, the RoPE part Rc is key only, and each row's f32 scale is
// hoisted out of its dot product; closing note: split-T kernels for long caches.
// Per (sequence b, head h):
//   z_t = sm * ( sLc_t <q_lat, dec(Lc_t)> + sRc_t <q_rope, dec(Rc_t)> )
//   o   = sum_t softmax(z)_t sLc_t dec(Lc_t)
//
// One CTA = one work item (sequence, group of N heads, range of tiles); N in
// {16, 32, 64}.
// The two contractions of a 128-token tile run on the tensor cores with fp16
// operands and f32 accumulators in TMEM; the per-row scales stay outside the MMA:
//   S^T[t][h] = K_t . Q_h      M = 128 tokens, N heads, K = 512 (S_L) and 64 (S_R)
//   z[t][h]   = c_h (sLc_t S_L + sRc_t S_R)                  (softmax warps)
//   P'[h][t]  = 2^(z - m_h) * sLc_t / s_ref                   (fp16, K-major in smem)
//   O^T[d][h] += sum_t V[t][d] P'[h][t]   M = 128 latent rows (x4), N heads, K = 128 tokens
// The e4m3 codes convert exactly to fp16.  One fp16 chunk of 128 tokens x 64
// channels (128-byte swizzle, K-major) feeds the score MMA as A, and two such
// chunks side by side feed the context MMA as an MN-major A operand, so Lc is
// converted twice per tile (once for each contraction) but never held whole.
//
// Warp roles (13 warps):
//   warp 0      issues every tcgen05.mma (lane 0 alone, or for N = 16 the whole
//               warp with one elected lane); the warp owns TMEM.
//   warps 1-8   softmax, two groups of four warps; a thread owns one token row
//               (its TMEM lane) and half of the heads: tile max per head by a
//               transposed warp reduction, running denominators per thread, lazy
//               rescaling of O (only when a head's max grows by more than 2^8).
//   warps 9-12  converters: warp w converts every 4th 16 KB chunk, alternating
//               between ring slots w and w+4 (e4m3 -> fp16 by the hardware cvt,
//               swizzled 16-byte stores), with the loads of its next chunk in
//               flight while it waits; the bulk-copy engine prefetches tiles into
//               L2 ahead of them.
// Chunk stream (converters and MMA in the same order): S(0), S(1), V(0), S(2),
// V(1), ..., V(n-1).  S(i) = Lc chunks 0..7, the Rc chunk and one empty pad
// chunk (so every V chunk pair lands on an even slot); V(i) = Lc chunks 0..7.
// The scores of tile i+1 run on the tensor cores while the softmax of tile i
// runs on the CUDA cores.  Every wait is bounded (2 s): on a timeout the CTA
// flags the workspace error word, drains its MMAs, frees TMEM and exits.
#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

using namespace ptx;

constexpr int RING = 8;                      // fp16 chunk slots, two per converter warp
constexpr int CHUNK = TILE * 64 * 2;         // 16 KB: 128 rows x 64 fp16
constexpr int S_CHUNKS = 10;                 // Lc 0..7, Rc, pad
constexpr int V_CHUNKS = 8;
constexpr int PERIOD = S_CHUNKS + V_CHUNKS;
constexpr int NCONV = 4;
constexpr int NSOFT = 8;
constexpr int WARP_SOFT = 1;
constexpr int WARP_CONV = WARP_SOFT + NSOFT;
constexpr int NTHREADS = (WARP_CONV + NCONV) * 32;
constexpr int L2_AHEAD = 3;                  // tiles prefetched into L2 ahead of the converters
constexpr float TAU = 8.0f;                  // rescale O only if a max grows by > 2^8
constexpr float TAU_S_POW = 64.0f;           // ... or the scale reference by > 2^6
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on any single wait
constexpr float LOG2E = 1.4426950408889634f;

constexpr int align1k(int x) { return (x + 1023) & ~1023; }

template <int N>
struct Lay {
  static constexpr int NH = N / 2;                         // heads per softmax group
  static constexpr int Q = 0;                              // 9 chunks [N x 64] fp16
  static constexpr int RINGO = align1k(Q + 9 * N * 128);
  static constexpr int P = RINGO + RING * CHUNK;           // 2 chunks [N x 64 tokens]
  static constexpr int BAR = P + 2 * N * 128;              // 32 mbarriers
  static constexpr int FLAGS = BAR + 32 * 8;               // tmem base, abort, corr flags
  static constexpr int CS = FLAGS + 32;                    // score constant per head
  static constexpr int MU = CS + N * 4;                    // max in use per head (log2)
  static constexpr int ALPHA = MU + N * 4;                 // rescale of l this tile
  static constexpr int FCOL = ALPHA + N * 4;               // rescale of O columns this tile
  static constexpr int LFIN = FCOL + N * 4;                // final denominators
  static constexpr int RMAX = LFIN + N * 4;                // [4][N] per-warp tile maxima
  static constexpr int RS = RMAX + 4 * N * 4;              // [2][4] warp max of sLc
  static constexpr int TOTAL = RS + 32;
  static constexpr int TMEM_COLS = (8 * N <= 128) ? 128 : (8 * N <= 256 ? 256 : 512);
};

// barrier indices
constexpr int B_FULL = 0, B_EMPTY = 8, B_S_FULL = 16, B_S_EMPTY = 18, B_P_FULL = 20,
              B_O_DONE = 21, B_G = 22 /* [group][2] */, B_DRAIN = 26;

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

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Offset of 16-byte unit u of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

// Position of flat chunk j in the stream S(0), S(1), V(0), S(2), V(1), ..., V(n-1).
struct ChunkInfo {
  int tile, c;  // c: 0..7 Lc channel block, 8 Rc, 9 pad
  bool v;
};
__device__ __forceinline__ ChunkInfo chunk_info(int j, int n_tiles) {
  if (j < S_CHUNKS) return {0, j, false};
  const int jj = j - S_CHUNKS, pair = jj / PERIOD, r = jj % PERIOD;
  if (pair < n_tiles - 1) {
    if (r < S_CHUNKS) return {pair + 1, r, false};
    return {pair, r - S_CHUNKS, true};
  }
  return {n_tiles - 1, r, true};
}
__device__ __forceinline__ int s_base(int i) { return i == 0 ? 0 : S_CHUNKS + PERIOD * (i - 1); }
__device__ __forceinline__ int v_base(int i, int n) {
  return i < n - 1 ? 2 * S_CHUNKS + PERIOD * i : S_CHUNKS + PERIOD * (n - 1);
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
__global__ void __launch_bounds__(NTHREADS, 1) decode_tc_kernel(const DecodeArgs a) {
  using L = Lay<N>;
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
  const int total_chunks = PERIOD * n_tiles;
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
    for (int i = 0; i < RING; ++i) {
      mbar_init(&bars[B_FULL + i], 1);
      mbar_init(&bars[B_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], NSOFT);
    }
    mbar_init(&bars[B_P_FULL], NSOFT);
    mbar_init(&bars[B_O_DONE], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_G + i], NSOFT / 2);
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) corr_flag[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < N) mu_s[threadIdx.x] = -INFINITY;
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
  const uint32_t ring_base = smem_u32(sm + L::RINGO);
  const uint32_t p_base = smem_u32(sm + L::P);
  const uint32_t q_base = smem_u32(sm + L::Q);

  if (warp == 0) {
    // ---------------------------------------------------------- MMA issuer
    // Narrow head groups (light softmax) issue from the whole converged warp with
    // elect.sync; wider ones from lane 0 alone, which leaves more issue slots on
    // this SM sub-partition to the softmax warps that share it (measured both
    // ways on the workloads of each width).
    constexpr bool WARP_ISSUE = (N <= 16);
    if (WARP_ISSUE || lane == 0) {
      const uint32_t idS = idesc_f16(128, N, false, false);
      const uint32_t idV = idesc_f16(128, N, true, false);
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
      auto wait_full = [&](int j) -> bool {
        const bool ok = wait(&bars[B_FULL + (j % RING)], (j / RING) & 1);
        tc_fence_after();
        return ok;
      };
      // Within a tile the loops run straight through; a failed wait only marks
      // the tile bad (the abort flag then makes every later wait return at once).
      auto issue_S = [&](int i) -> bool {
        const int buf = i & 1;
        if (!wait(&bars[B_S_EMPTY + buf], ((i >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const uint32_t dL = tmem + buf * 2 * N, dR = dL + N;
        const int base = s_base(i);
        bool good = true;
        for (int c = 0; c < 9; ++c) {
          const int j = base + c;
          good = wait_full(j) && good;
          const uint32_t ab = ring_base + (j % RING) * CHUNK, bb = q_base + c * N * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma(c < 8 ? dL : dR, smem_desc(ab + kk * 32, 16, 1024, SW128),
                smem_desc(bb + kk * 32, 16, 1024, SW128), idS, (c == 8 ? kk : (c | kk)) != 0);
          commit(&bars[B_EMPTY + (j % RING)]);
        }
        // the pad chunk carries no data: hand its slot straight back
        good = wait_full(base + 9) && good;
        if (!good) return false;
        if (!WARP_ISSUE || lane == 0) mbar_arrive(&bars[B_EMPTY + ((base + 9) % RING)]);
        commit(&bars[B_S_FULL + buf]);
        return true;
      };
      auto issue_V = [&](int i) -> bool {
        if (!wait(&bars[B_P_FULL], i & 1)) return false;
        tc_fence_after();
        const int base = v_base(i, n_tiles);
        bool good = true;
        for (int m = 0; m < 4; ++m) {
          const int j = base + 2 * m;  // slot j % RING is even, j + 1 is the next slot
          good = wait_full(j) && good;
          good = wait_full(j + 1) && good;
          const uint32_t ab = ring_base + (j % RING) * CHUNK;
          const uint32_t d = tmem + 4 * N + m * N;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A = V^T: MN-major, 64-channel atoms CHUNK bytes apart, 8-token groups 1 KB apart
            const uint64_t ad = smem_desc(ab + kk * 2048, CHUNK, 1024, SW128);
            const uint64_t bd =
                smem_desc(p_base + (kk >> 2) * N * 128 + (kk & 3) * 32, 16, 1024, SW128);
            mma(d, ad, bd, idV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          commit(&bars[B_EMPTY + (j % RING)]);
          commit(&bars[B_EMPTY + ((j + 1) % RING)]);
        }
        if (!good) return false;
        commit(&bars[B_O_DONE]);
        return true;
      };
      bool ok = issue_S(0);
      for (int i = 1; ok && i < n_tiles; ++i) ok = issue_S(i) && issue_V(i - 1);
      if (ok) ok = issue_V(n_tiles - 1);
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
    auto group_sync = [&](int k, int i) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_G + 2 * grp + k]);
      return mbar_wait_warp(&bars[B_G + 2 * grp + k], i & 1, abort_flag, WAIT_NS);
    };
    // P'[h][t] element address (K-major [N x 64] chunks, token chunk = row >> 6)
    const uint32_t prow = p_base + (row >> 6) * N * 128;
    const int tcol = row & 63;
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
      float z[NH];
#pragma unroll
      for (int c = 0; c < NH; c += 8) {
        uint32_t rl[8], rr[8];
        tmem_ld8(tmem + lane_addr + buf * 2 * N + hb + c, rl);
        tmem_ld8(tmem + lane_addr + buf * 2 * N + N + hb + c, rr);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          z[c + j] = valid ? cs[hb + c + j] * (sL * __uint_as_float(rl[j]) +
                                               sR * __uint_as_float(rr[j]))
                           : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_EMPTY + buf]);

      // tile max per head (and of sLc) over the group's four warps
      {
        const float mx = warp_transpose_reduce<NH, true>(z, lane);
        if ((lane & ((32 >> LOG2_NH) - 1)) == 0)
          rmax[wq * N + hb + (lane >> (5 - LOG2_NH))] = mx;
        float smax = valid ? sL : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) rs[grp * 4 + wq] = smax;
      }
      if (!group_sync(0, i)) { ok = false; break; }
      const float smax = fmaxf(fmaxf(rs[grp * 4 + 0], rs[grp * 4 + 1]),
                               fmaxf(rs[grp * 4 + 2], rs[grp * 4 + 3]));
      const float sref_new = (smax > sref * TAU_S_POW) ? smax : sref;
      const float beta = (sref_new == sref) ? 1.f : (sref > 0.f ? sref / sref_new : 0.f);
      if (st == 0) corr_flag[grp * 2 + ((i + 1) & 1)] = 0;  // flag of the next tile
      if (st < NH) {
        const int hh = hb + st;
        const float tmax = fmaxf(fmaxf(rmax[hh], rmax[N + hh]), fmaxf(rmax[2 * N + hh], rmax[3 * N + hh]));
        float mu = mu_s[hh];
        const float mn = fmaxf(mu, tmax);
        float alpha = 1.f;
        if (mn > mu + TAU) {
          alpha = (mu == -INFINITY) ? 0.f : ex2_approx(mu - mn);
          mu = mn;
        }
        mu_s[hh] = mu;
        alpha_s[hh] = alpha;
        fcol[hh] = alpha * beta;
        if (i > 0 && alpha * beta != 1.f) corr_flag[grp * 2 + (i & 1)] = 1;
      }
      sref = sref_new;
      if (!group_sync(1, i)) { ok = false; break; }

      // probabilities; running denominators; fp16 P' = p * sLc / s_ref
      const float w = valid ? sL * (sref > 0.f ? 1.0f / sref : 0.f) : 0.f;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float p = (z[h] == -INFINITY) ? 0.f : ex2_approx(z[h] - mu_s[hb + h]);
        lpart[h] = lpart[h] * alpha_s[hb + h] + p;
        z[h] = p * w;
      }
      if (i > 0) {
        if (!mbar_wait_warp(&bars[B_O_DONE], (i - 1) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (corr_flag[grp * 2 + (i & 1)]) {
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int c = 0; c < NH; c += 8) {
              uint32_t r[8];
              const uint32_t ad = tmem + lane_addr + 4 * N + m * N + hb + c;
              tmem_ld8(ad, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 8; ++j)
                r[j] = __float_as_uint(__uint_as_float(r[j]) * fcol[hb + c + j]);
              tmem_st8(ad, r);
            }
          }
          tmem_wait_st();
        }
      }
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int hr = hb + h;
        sts16(prow + sw128(hr, tcol >> 3) + (tcol & 7) * 2, __half_as_ushort(__float2half_rn(z[h])));
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
      if (group_sync(0, n_tiles)) {
        if (st < NH) {
          const int hh = hb + st;
          lfin[hh] = (rmax[hh] + rmax[N + hh]) + (rmax[2 * N + hh] + rmax[3 * N + hh]);
        }
        if (group_sync(1, n_tiles)) {
          // epilogue: unnormalised partial o = acc * s_ref, with (m, l) per head
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
                  a.ws_o[(base + h) * DL + m * 128 + row] = __uint_as_float(r[j]) * sref;
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
    // Warp cw converts chunks j = cw, cw + 4, ... into ring slot j % 8.  Lane l
    // handles rows 8i + (l >> 2) (i = 0..15) and 16-byte piece (l & 3) of the
    // chunk's 64 bytes per row; rows 0..63 are the tile's first page, 64..127 its
    // second.
    const int cw = warp - WARP_CONV;
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
    uint4 dat[16];
    auto load = [&](int j) {
      const ChunkInfo ci = chunk_info(j, n_tiles);
      if (ci.c == 9) return;  // pad chunk
      const uint8_t *p0, *p1;
      int nv;
      pages_of(ci.tile, p0, p1, nv);
      const int off = ci.c * 64 + sub * 16;  // c == 8 is the Rc block: channels 512..575
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 8 * i + rin;
        const uint8_t* pg = (i < 8) ? p0 : p1;
        dat[i] = (pg != nullptr && r < nv) ? ldg16(pg + (size_t)(r & 63) * D + off)
                                           : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    bool ok = true;
    if (cw == 0 && lane == 0) {
      // the first tiles' lines: ask the bulk-copy engine for them up front
      for (int tl = 0; tl < L2_AHEAD && tl < n_tiles; ++tl) {
        for (int pg = 0; pg < 2; ++pg) {
          const int64_t tk = t0 + (int64_t)tl * TILE + pg * PAGE;
          if (tk >= t_end) break;
          const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
          const int64_t slot = slot_of(a, b, tk);
          if (slot >= 0) prefetch_l2(a.codes + slot * D, (uint32_t)(nt * D));
        }
      }
    }
    if (cw < total_chunks) load(cw);
    for (int j = cw; j < total_chunks && ok; j += NCONV) {
      const ChunkInfo ci = chunk_info(j, n_tiles);
      const int slot = j % RING;
      const uint32_t slot_addr = ring_base + slot * CHUNK;
      if (!mbar_wait_warp(&bars[B_EMPTY + slot], ((j / RING) & 1) ^ 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      if (ci.c != 9) {
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
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_FULL + slot]);
      if (j + NCONV < total_chunks) load(j + NCONV);
      // L2 prefetch of the tile L2_AHEAD tiles ahead, by whoever converts its S(i) chunk 0
      if (lane == 0 && !ci.v && ci.c == 0 && ci.tile + L2_AHEAD < n_tiles) {
        const int64_t tb = t0 + (int64_t)(ci.tile + L2_AHEAD) * TILE;
        for (int pg = 0; pg < 2; ++pg) {
          const int64_t tk = tb + pg * PAGE;
          if (tk >= t_end) break;
          const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
          const int64_t slot = slot_of(a, b, tk);
          if (slot >= 0) prefetch_l2(a.codes + slot * D, (uint32_t)(nt * D));
        }
      }
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
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  decode_tc_kernel<N><<<a.plan.max_items, NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

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
