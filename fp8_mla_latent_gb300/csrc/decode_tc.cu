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
// One CTA = one (split of T, group of N heads, sequence); N in {16, 32, 64}.
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
//   warp 0      one thread issues every tcgen05.mma; the warp owns TMEM.
//   warps 1-4   softmax: thread <-> TMEM lane <-> token row of the tile; tile
//               max / sum per head by warp transposed reductions, lazy rescaling
//               of O (only when a head's max grows by more than 2^8).
//   warps 5-12  converters: 16-byte global loads of e4m3 rows (six chunks ahead
//               in registers; the bulk-copy engine prefetches tiles into L2),
//               exact cvt to fp16, swizzled 16-byte stores into a 6-slot ring.
// MMA issue order is S(0), S(1), V(0), S(2), V(1), ...: the scores of tile i+1
// run on the tensor cores while the softmax of tile i runs on the CUDA cores.
// Every wait is bounded (2 s): on a timeout the CTA flags the workspace error
// word, drains its MMAs, frees TMEM and exits.
#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

using namespace ptx;

constexpr int RING = 6;                      // fp16 Lc chunk slots (even: pairs never wrap)
constexpr int RC_SLOTS = 2;
constexpr int CHUNK = TILE * 64 * 2;         // 16 KB: 128 rows x 64 fp16
constexpr int NCONV = 8;
constexpr int CONV_DEPTH = 6;               // chunks of e4m3 loads in flight per converter
constexpr int L2_AHEAD = 3;                 // tiles prefetched into L2 ahead of the converters
constexpr int NSOFT = 4;
constexpr int WARP_SOFT = 1;
constexpr int WARP_CONV = WARP_SOFT + NSOFT;
constexpr int NTHREADS = (WARP_CONV + NCONV) * 32;
constexpr float TAU = 8.0f;                  // rescale O only if a max grows by > 2^8
constexpr float TAU_S_POW = 64.0f;           // ... or the scale reference by > 2^6
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on any single wait
constexpr float LOG2E = 1.4426950408889634f;

constexpr int align1k(int x) { return (x + 1023) & ~1023; }

template <int N>
struct Lay {
  static constexpr int Q = 0;                              // 9 chunks [N x 64] fp16
  static constexpr int RINGO = align1k(Q + 9 * N * 128);
  static constexpr int RCO = RINGO + RING * CHUNK;
  static constexpr int P = RCO + RC_SLOTS * CHUNK;         // 2 chunks [N x 64 tokens]
  static constexpr int BAR = P + 2 * N * 128;              // 32 mbarriers
  static constexpr int FLAGS = BAR + 32 * 8;               // tmem base, abort, need_corr
  static constexpr int CS = FLAGS + 16;                    // score constant per head
  static constexpr int MU = CS + N * 4;                    // max in use per head (log2)
  static constexpr int LACC = MU + N * 4;                  // softmax denominator per head
  static constexpr int ALPHA = LACC + N * 4;               // rescale of l this tile
  static constexpr int FCOL = ALPHA + N * 4;               // rescale of O columns this tile
  static constexpr int RMAX = FCOL + N * 4;                // [4][N] warp maxima
  static constexpr int RSUM = RMAX + 4 * N * 4;            // [4][N] warp sums
  static constexpr int RS = RSUM + 4 * N * 4;              // [4] warp max of sLc
  static constexpr int TOTAL = RS + 16;
  static constexpr int TMEM_COLS = (8 * N <= 128) ? 128 : (8 * N <= 256 ? 256 : 512);
};

// barrier indices
constexpr int B_RING_FULL = 0, B_RING_EMPTY = 6, B_RC_FULL = 12, B_RC_EMPTY = 14, B_S_FULL = 16,
              B_S_EMPTY = 18, B_P_FULL = 20, B_O_DONE = 21, B_G0 = 22, B_DRAIN = 25;

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

// Offset of 16-byte unit u of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

// Position of flat chunk j in the converter/MMA order S(0), S(1), V(0), S(2), V(1), ...
// S(i) has 9 chunks (Lc 0..7, then Rc), V(i) has 8 (Lc 0..7).
struct ChunkInfo {
  int tile, c;
  bool v;
};
__device__ __forceinline__ ChunkInfo chunk_info(int j, int n_tiles) {
  if (j < 9) return {0, j, false};
  const int jj = j - 9, pair = jj / 17, r = jj % 17;
  if (pair < n_tiles - 1) {
    if (r < 9) return {pair + 1, r, false};
    return {pair, r - 9, true};
  }
  return {n_tiles - 1, jj - 17 * (n_tiles - 1), true};
}

// Transposed warp reduction: lane holds v[0..N); afterwards lane holds the
// reduction over all 32 lanes of heads h = lane*(N/32) + j (N >= 32), or of
// head lane>>1 in out[0] (N == 16).
template <int N, bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(const float (&v)[N], float* out,
                                                      int lane) {
  float t[N / 2];
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int j = 0; j < N / 2; ++j) {
      const float send = up ? v[j] : v[j + N / 2];
      const float keep = up ? v[j + N / 2] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      t[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  int n = N / 2;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < N / 4; ++j) {
        if (j < n / 2) {
          const float send = up ? t[j] : t[j + n / 2];
          const float keep = up ? t[j + n / 2] : t[j];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          t[j] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
      }
      n >>= 1;
    } else {
      // one value left per lane and a lane bit still unreduced (N == 16 only)
      const float recv = __shfl_xor_sync(0xffffffffu, t[0], o);
      t[0] = MAX ? fmaxf(t[0], recv) : t[0] + recv;
    }
  }
#pragma unroll
  for (int j = 0; j < (N >= 32 ? N / 32 : 1); ++j) out[j] = t[j];
}

template <int N>
__global__ void __launch_bounds__(NTHREADS, 1) decode_tc_kernel(const DecodeArgs a) {
  using L = Lay<N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t T = seq_len_of(a, b);
  const int64_t split_len = (int64_t)a.plan.split_tiles * TILE;
  const int64_t t0 = (int64_t)split * split_len;
  if (t0 >= T) return;  // empty split: the combine kernel skips it
  const int64_t t_end = (t0 + split_len < T) ? t0 + split_len : T;
  const int n_tiles = (int)((t_end - t0 + TILE - 1) / TILE);
  const int h0 = g * N;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::FLAGS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::FLAGS + 4);
  volatile int* need_corr = reinterpret_cast<volatile int*>(sm + L::FLAGS + 8);
  float* cs = reinterpret_cast<float*>(sm + L::CS);
  float* mu_s = reinterpret_cast<float*>(sm + L::MU);
  float* lacc = reinterpret_cast<float*>(sm + L::LACC);
  float* alpha_s = reinterpret_cast<float*>(sm + L::ALPHA);
  float* fcol = reinterpret_cast<float*>(sm + L::FCOL);
  float* rmax = reinterpret_cast<float*>(sm + L::RMAX);
  float* rsum = reinterpret_cast<float*>(sm + L::RSUM);
  float* rs = reinterpret_cast<float*>(sm + L::RS);

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < RING; ++i) {
      mbar_init(&bars[B_RING_FULL + i], NCONV);
      mbar_init(&bars[B_RING_EMPTY + i], 1);
    }
    for (int i = 0; i < RC_SLOTS; ++i) {
      mbar_init(&bars[B_RC_FULL + i], NCONV);
      mbar_init(&bars[B_RC_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_S_EMPTY + i], NSOFT);
    }
    mbar_init(&bars[B_P_FULL], NSOFT);
    mbar_init(&bars[B_O_DONE], 1);
    for (int i = 0; i < 3; ++i) mbar_init(&bars[B_G0 + i], NSOFT);
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    *need_corr = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < N) {
    mu_s[threadIdx.x] = -INFINITY;
    lacc[threadIdx.x] = 0.f;
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
  const uint32_t ring_base = smem_u32(sm + L::RINGO);
  const uint32_t rc_base = smem_u32(sm + L::RCO);
  const uint32_t p_base = smem_u32(sm + L::P);
  const uint32_t q_base = smem_u32(sm + L::Q);

  if (warp == 0) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_f16(128, N, false, false);
      const uint32_t idV = idesc_f16(128, N, true, false);
      uint32_t k = 0;  // Lc ring chunk counter
      bool ok = true;
      auto issue_S = [&](int i) -> bool {
        const int buf = i & 1;
        if (!mbar_wait(&bars[B_S_EMPTY + buf], ((i >> 1) & 1) ^ 1, abort_flag, WAIT_NS))
          return false;
        tc_fence_after();
        const uint32_t dL = tmem + buf * 2 * N, dR = dL + N;
        for (int c = 0; c < 8; ++c, ++k) {
          const int slot = k % RING;
          if (!mbar_wait(&bars[B_RING_FULL + slot], (k / RING) & 1, abort_flag, WAIT_NS))
            return false;
          tc_fence_after();
          const uint32_t ab = ring_base + slot * CHUNK, bb = q_base + c * N * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(dL, smem_desc(ab + kk * 32, 16, 1024, SW128),
                    smem_desc(bb + kk * 32, 16, 1024, SW128), idS, (c | kk) != 0);
          mma_commit(&bars[B_RING_EMPTY + slot]);
        }
        const int rsl = i % RC_SLOTS;
        if (!mbar_wait(&bars[B_RC_FULL + rsl], (i / RC_SLOTS) & 1, abort_flag, WAIT_NS))
          return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(dR, smem_desc(rc_base + rsl * CHUNK + kk * 32, 16, 1024, SW128),
                  smem_desc(q_base + 8 * N * 128 + kk * 32, 16, 1024, SW128), idS, kk != 0);
        mma_commit(&bars[B_RC_EMPTY + rsl]);
        mma_commit(&bars[B_S_FULL + buf]);
        return true;
      };
      auto issue_V = [&](int i) -> bool {
        if (!mbar_wait(&bars[B_P_FULL], i & 1, abort_flag, WAIT_NS)) return false;
        tc_fence_after();
        for (int m = 0; m < 4; ++m, k += 2) {
          const int slot = k % RING;  // even
          if (!mbar_wait(&bars[B_RING_FULL + slot], (k / RING) & 1, abort_flag, WAIT_NS))
            return false;
          if (!mbar_wait(&bars[B_RING_FULL + slot + 1], (k / RING) & 1, abort_flag, WAIT_NS))
            return false;
          tc_fence_after();
          const uint32_t ab = ring_base + slot * CHUNK;
          const uint32_t d = tmem + 4 * N + m * N;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A = V^T: MN-major, 64-channel atoms CHUNK bytes apart, 8-token groups 1 KB apart
            const uint64_t ad = smem_desc(ab + kk * 2048, CHUNK, 1024, SW128);
            const uint64_t bd =
                smem_desc(p_base + (kk >> 2) * N * 128 + (kk & 3) * 32, 16, 1024, SW128);
            mma_f16(d, ad, bd, idV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars[B_RING_EMPTY + slot]);
          mma_commit(&bars[B_RING_EMPTY + slot + 1]);
        }
        mma_commit(&bars[B_O_DONE]);
        return true;
      };
      ok = issue_S(0);
      for (int i = 1; ok && i < n_tiles; ++i) ok = issue_S(i) && issue_V(i - 1);
      if (ok) ok = issue_V(n_tiles - 1);
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.err, ERR_TIMEOUT);
      }
      // drain: every MMA issued above completes before TMEM is released
      const int zero = 0;
      mma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
    }
    __syncwarp();
  } else if (warp < WARP_CONV) {
    // ---------------------------------------------------------- softmax
    const int st = threadIdx.x - WARP_SOFT * 32;  // 0..127
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;          // TMEM lane = token row of the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int wq = warp - WARP_SOFT;              // 0..3 slot in the reduction arrays
    float sref = 0.f;
    bool ok = true;
    auto group_sync = [&](int id, int i) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_G0 + id]);
      return mbar_wait(&bars[B_G0 + id], i & 1, abort_flag, WAIT_NS);
    };
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
      if (!mbar_wait(&bars[B_S_FULL + buf], (i >> 1) & 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float z[N];
#pragma unroll
      for (int c = 0; c < N; c += 16) {
        uint32_t rl[16], rr[16];
        tmem_ld16(tmem + lane_addr + buf * 2 * N + c, rl);
        tmem_ld16(tmem + lane_addr + buf * 2 * N + N + c, rr);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          z[c + j] = valid ? cs[c + j] * (sL * __uint_as_float(rl[j]) + sR * __uint_as_float(rr[j]))
                           : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_EMPTY + buf]);

      // tile max per head and of sLc
      {
        float mx[N >= 32 ? N / 32 : 1];
        warp_transpose_reduce<N, true>(z, mx, lane);
        if (N >= 32) {
#pragma unroll
          for (int j = 0; j < (N >= 32 ? N / 32 : 1); ++j) rmax[wq * N + lane * (N / 32) + j] = mx[j];
        } else if ((lane & 1) == 0) {
          rmax[wq * N + (lane >> 1)] = mx[0];
        }
        float smax = valid ? sL : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) rs[wq] = smax;
      }
      if (!group_sync(0, i)) { ok = false; break; }
      const float smax = fmaxf(fmaxf(rs[0], rs[1]), fmaxf(rs[2], rs[3]));
      const float sref_new = (smax > sref * TAU_S_POW) ? smax : sref;
      const float beta = (sref_new == sref) ? 1.f : (sref > 0.f ? sref / sref_new : 0.f);
      if (st < N) {
        const float tmax = fmaxf(fmaxf(rmax[st], rmax[N + st]), fmaxf(rmax[2 * N + st], rmax[3 * N + st]));
        float mu = mu_s[st];
        const float mn = fmaxf(mu, tmax);
        float alpha = 1.f;
        if (mn > mu + TAU) {
          alpha = (mu == -INFINITY) ? 0.f : exp2f(mu - mn);
          mu = mn;
        }
        mu_s[st] = mu;
        alpha_s[st] = alpha;
        fcol[st] = alpha * beta;
        if (i > 0 && alpha * beta != 1.f) *need_corr = 1;
      }
      sref = sref_new;
      if (!group_sync(1, i)) { ok = false; break; }

      // probabilities, tile sums, fp16 P'
#pragma unroll
      for (int h = 0; h < N; ++h) z[h] = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - mu_s[h]);
      {
        float sm_[N >= 32 ? N / 32 : 1];
        warp_transpose_reduce<N, false>(z, sm_, lane);
        if (N >= 32) {
#pragma unroll
          for (int j = 0; j < (N >= 32 ? N / 32 : 1); ++j) rsum[wq * N + lane * (N / 32) + j] = sm_[j];
        } else if ((lane & 1) == 0) {
          rsum[wq * N + (lane >> 1)] = sm_[0];
        }
      }
      const float w = valid ? sL * (sref > 0.f ? 1.0f / sref : 0.f) : 0.f;
      if (i > 0) {
        if (!mbar_wait(&bars[B_O_DONE], (i - 1) & 1, abort_flag, WAIT_NS)) { ok = false; break; }
        tc_fence_after();
        if (*need_corr) {
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int c = 0; c < N; c += 16) {
              uint32_t r[16];
              const uint32_t ad = tmem + lane_addr + 4 * N + m * N + c;
              tmem_ld16(ad, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * fcol[c + j]);
              tmem_st16(ad, r);
            }
          }
          tmem_wait_st();
        }
      }
      // P'[h][t] as fp16, K-major [N x 128 tokens]: lanes t, t^1 swap halves so each
      // writes one 32-bit word {P'[h][t_even], P'[h][t_even+1]}.
      {
        const uint32_t pchunk = p_base + (row >> 6) * N * 128;
        const int tcol = row & 63;
        const bool odd = (lane & 1) != 0;
#pragma unroll
        for (int h = 0; h < N; h += 2) {
          const __half2 mine = __floats2half2_rn(z[h] * w, z[h + 1] * w);
          const uint32_t mw = *reinterpret_cast<const uint32_t*>(&mine);
          const uint32_t other = __shfl_xor_sync(0xffffffffu, mw, 1);
          // even lane: {mine.lo, other.lo} for head h; odd lane: {other.hi, mine.hi} for head h+1
          const uint32_t word = odd ? __byte_perm(other, mw, 0x7632) : __byte_perm(mw, other, 0x5410);
          const int hr = odd ? h + 1 : h;
          const int tc = tcol & ~1;
          const uint32_t ad = pchunk + sw128(hr, tc >> 3) + (tc & 7) * 2;
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(ad), "r"(word) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P_FULL]);
      if (!group_sync(2, i)) { ok = false; break; }
      if (st < N)
        lacc[st] = lacc[st] * alpha_s[st] +
                   ((rsum[st] + rsum[N + st]) + (rsum[2 * N + st] + rsum[3 * N + st]));
      if (st == 0) *need_corr = 0;
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    } else if (mbar_wait(&bars[B_O_DONE], (n_tiles - 1) & 1, abort_flag, WAIT_NS)) {
      // epilogue: unnormalised partial o = acc * s_ref, with (m, l) per head
      tc_fence_after();
      const int64_t base = ((int64_t)b * a.plan.n_splits + split) * a.H + h0;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int c = 0; c < N; c += 16) {
          uint32_t r[16];
          tmem_ld16(tmem + lane_addr + 4 * N + m * N + c, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (h0 + c + j < a.H)
              a.ws_o[(base + c + j) * DL + m * 128 + row] = __uint_as_float(r[j]) * sref;
        }
      }
      if (st < N && h0 + st < a.H) {
        a.ws_m[base + st] = mu_s[st];
        a.ws_l[base + st] = lacc[st];
      }
    } else {
      *abort_flag = 1;
      atomicOr(a.err, ERR_TIMEOUT);
    }
  } else {
    // ---------------------------------------------------------- converters
    const int ct = threadIdx.x - WARP_CONV * 32;  // 0..255
    const int r0 = ct >> 2, sub = ct & 3;         // rows r0 and r0 + 64, 16-byte piece `sub`
    const int total = 17 * n_tiles;
    int ctile[2] = {-1, -1};
    const uint8_t* cptr[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
    auto rows_of = [&](int tile, const uint8_t*& p0, const uint8_t*& p1) {
      if (ctile[0] == tile) { p0 = cptr[0][0]; p1 = cptr[0][1]; return; }
      if (ctile[1] == tile) { p0 = cptr[1][0]; p1 = cptr[1][1]; return; }
      const uint8_t* q[2];
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int64_t tok = t0 + (int64_t)tile * TILE + r0 + 64 * k2;
        q[k2] = nullptr;
        if (tok < t_end) {
          const int64_t slot = slot_of(a, b, tok);
          if (slot >= 0) q[k2] = a.codes + slot * D + sub * 16;
        }
      }
      ctile[1] = ctile[0]; cptr[1][0] = cptr[0][0]; cptr[1][1] = cptr[0][1];
      ctile[0] = tile; cptr[0][0] = q[0]; cptr[0][1] = q[1];
      p0 = q[0]; p1 = q[1];
    };
    auto load = [&](int j, uint4& x0, uint4& x1) {
      const ChunkInfo ci = chunk_info(j, n_tiles);
      const uint8_t *p0, *p1;
      rows_of(ci.tile, p0, p1);
      const int dim0 = ci.c * 64;  // c == 8 is the Rc chunk: channels 512..575
      x0 = p0 ? ldg16(p0 + dim0) : make_uint4(0u, 0u, 0u, 0u);
      x1 = p1 ? ldg16(p1 + dim0) : make_uint4(0u, 0u, 0u, 0u);
    };
    // CONV_DEPTH chunks of loads stay in flight per thread (8 KB per chunk per CTA)
    uint4 R[CONV_DEPTH][2];
    uint32_t k = 0;
    bool ok = true;
    auto convert_store = [&](uint32_t dst, int r, const uint4& x) {
      uint32_t h[8];
      h[0] = e4m3x2_to_f16x2((uint16_t)(x.x & 0xFFFFu)); h[1] = e4m3x2_to_f16x2((uint16_t)(x.x >> 16));
      h[2] = e4m3x2_to_f16x2((uint16_t)(x.y & 0xFFFFu)); h[3] = e4m3x2_to_f16x2((uint16_t)(x.y >> 16));
      h[4] = e4m3x2_to_f16x2((uint16_t)(x.z & 0xFFFFu)); h[5] = e4m3x2_to_f16x2((uint16_t)(x.z >> 16));
      h[6] = e4m3x2_to_f16x2((uint16_t)(x.w & 0xFFFFu)); h[7] = e4m3x2_to_f16x2((uint16_t)(x.w >> 16));
      sts128(dst + sw128(r, 2 * sub), make_uint4(h[0], h[1], h[2], h[3]));
      sts128(dst + sw128(r, 2 * sub + 1), make_uint4(h[4], h[5], h[6], h[7]));
    };
    // convert chunk j (its codes are in cur), publish it, then refill cur with chunk j + CONV_DEPTH
    auto step = [&](int j, uint4 (&cur)[2]) -> bool {
      const ChunkInfo ci = chunk_info(j, n_tiles);
      uint64_t* full;
      uint32_t dst;
      if (ci.c == 8) {
        const int s = ci.tile % RC_SLOTS;
        if (!mbar_wait(&bars[B_RC_EMPTY + s], ((ci.tile / RC_SLOTS) & 1) ^ 1, abort_flag, WAIT_NS))
          return false;
        dst = rc_base + s * CHUNK;
        full = &bars[B_RC_FULL + s];
      } else {
        const int s = k % RING;
        if (!mbar_wait(&bars[B_RING_EMPTY + s], ((k / RING) & 1) ^ 1, abort_flag, WAIT_NS))
          return false;
        dst = ring_base + s * CHUNK;
        full = &bars[B_RING_FULL + s];
        ++k;
      }
      convert_store(dst, r0, cur[0]);
      convert_store(dst, r0 + 64, cur[1]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full);
      if (j + CONV_DEPTH < total) load(j + CONV_DEPTH, cur[0], cur[1]);
      // L2 prefetch of the tile L2_AHEAD tiles ahead, once per tile, by the bulk-copy engine
      if (ct == 0 && !ci.v && ci.c == 0 && ci.tile + L2_AHEAD < n_tiles) {
        const int64_t tb = t0 + (int64_t)(ci.tile + L2_AHEAD) * TILE;
        for (int pg = 0; pg < TILE / PAGE; ++pg) {
          const int64_t tk = tb + pg * PAGE;
          if (tk >= t_end) break;
          const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
          const int64_t slot = slot_of(a, b, tk);
          if (slot >= 0) prefetch_l2(a.codes + slot * D, (uint32_t)(nt * D));
        }
      }
      return true;
    };
    // the first tiles' lines: ask the bulk-copy engine for them before the loads below
    if (ct == 0) {
      for (int tl = 0; tl < L2_AHEAD && tl < n_tiles; ++tl) {
        for (int pg = 0; pg < TILE / PAGE; ++pg) {
          const int64_t tk = t0 + (int64_t)tl * TILE + pg * PAGE;
          if (tk >= t_end) break;
          const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
          const int64_t slot = slot_of(a, b, tk);
          if (slot >= 0) prefetch_l2(a.codes + slot * D, (uint32_t)(nt * D));
        }
      }
    }
#pragma unroll
    for (int d = 0; d < CONV_DEPTH; ++d)
      if (d < total) load(d, R[d][0], R[d][1]);
    for (int j0 = 0; j0 < total && ok; j0 += CONV_DEPTH) {
#pragma unroll
      for (int d = 0; d < CONV_DEPTH; ++d)
        if (ok && j0 + d < total) ok = step(j0 + d, R[d]);
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
  dim3 grid(a.plan.n_splits, a.plan.n_hg, a.B);
  decode_tc_kernel<N><<<grid, NTHREADS, smem, s>>>(a);
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
