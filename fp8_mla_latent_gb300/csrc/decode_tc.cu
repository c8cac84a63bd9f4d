// decode_tc.cu -- tcgen05 tensor-core split-T absorbed MLA decode over the e4m3
// latent cache, one CTA per SM, for groups of 16 or 32 heads.
//
// Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description: the latent Lc is both key and value of the
// absorbed attention, the RoPE part Rc is key only, and each row's f32 scale is
// applied outside its dot product; closing note: split-T kernels for long caches.
// Per (sequence b, head h):
//   z_t = sm * ( sLc_t <q_lat, dec(Lc_t)> + sRc_t <q_rope, dec(Rc_t)> )
//   o   = sum_t softmax(z)_t sLc_t dec(Lc_t)
//
// One CTA = one work item (sequence, group of N heads, range of 128-token tiles).
// When every (sequence, head group) pair holds at least a range's worth of tiles,
// the items are instead equal ranges of the tiles of all pairs in order, one per
// CTA: a range that reaches the end of its pair continues into the next one, as a
// second segment with its own query, page table and partial (the softmax warps put
// the next query in place as soon as they have seen the first segment's last
// scores, so the next scores overlap the first segment's epilogue).
// Every byte of a tile is loaded once, by TMA: the four Lc blocks into a ring of
// [128 tokens x 128 bytes] slots (128-byte swizzle), the Rc block into a ring of
// [128 tokens x 64 bytes] slots (64-byte swizzle).  Both contractions read those
// bytes as they are, with e4m3 operands and f32 accumulators in TMEM:
//   S[t][h]   = K_t . Q_h      kind::f8f6f4, M = 128 tokens, N = 2N' columns
//                              (the query's hi terms, then its lo terms: one MMA
//                              reads the tile once for both), K = 512 (S_L) and 64
//                              (S_R); A = the Lc / Rc block (K-major), B = the
//                              query prepared by the query-prep launch (two e4m3
//                              terms on one power-of-two scale per head)
//   z[t][h]   = c_h (sLc_t (S_L hi + S_L lo) + sRc_t (S_R hi + S_R lo))  (softmax warps)
//   P''[h][t] = 2^(z - m_h) (sLc_t / s_ref) P_TOP   as two e4m3 terms, hi + lo
//   O[d][h]  += sum_t V[t][d] P''[h][t]   kind::f8f6f4, M = 128 latent rows (x4
//                              d-blocks), N = 2N' (hi and lo weight columns), K =
//                              32 tokens; A = the same Lc block read MN-major
// The hi and lo columns of S and of O are added in f32 by the softmax and the
// epilogue.
//
// Warp roles (11 warps):
//   warp 0      loads the item's page table, then per tile the row scales, the Rc
//               block and the four Lc blocks by TMA (a block as soon as its ring
//               slot is free); it owns TMEM.  (An L2 prefetch of the tiles ahead
//               was measured: its bulk requests delay the loads behind them, and
//               the loop ran 10 % slower with it.)
//   warp 1      issues the score MMAs of each tile once its blocks are in and its
//               S buffer is free (S is double-buffered).
//   warp 2      zeroes the Lc rows that hold no data, then issues the context MMAs
//               of a tile once its P'' is written; each Lc block's slot is released
//               by the commit after its MMAs.
//   warps 3-10  softmax, two groups of four warps; a thread owns one token row (its
//               TMEM lane) and half of the heads: tile maximum per head by a
//               transposed warp reduction and one exchange per group and tile,
//               lazy running maxima kept by every thread of the group alike,
//               running denominators per thread, the O rescale of the heads whose
//               factor moved, P'' in shared memory (double-buffered).
// Every wait is bounded (2 s): on a timeout the CTA flags the workspace error
// word, drains its MMAs and its TMA loads, frees TMEM and exits.  Parity waits:
// no barrier is ever armed or completed two phases ahead of a thread that still
// waits on it (the ring and buffer sizes below keep that true).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

using namespace ptx;

constexpr int KBLK = TILE * 128;             // 16 KB: [128 tokens x 128 bytes] (an Lc block)
constexpr int RBLK = TILE * 64;              // 8 KB: [128 tokens x 64 bytes] (the Rc block)
constexpr int W_TMA = 0, W_MMA = 1, W_CTX = 2, W_SOFT = 3;
constexpr int NSOFT = 8;
constexpr int NTHREADS = (W_SOFT + NSOFT) * 32;
constexpr int NTF = 4;                       // tile-loaded barriers, scale slots, page facts
// Lazy rescaling thresholds.  The e4m3 weights P'' = 2^(z - m) (sLc / s_ref)
// P_TOP are at most 2^TAU * TAU_S * P_TOP = 256 <= 448, and with this little
// headroom the largest weights of a tile sit near the top of the e4m3 range,
// where the two-term split keeps about 8 significant bits.
constexpr float TAU = 1.0f;                  // move a head's max if a tile's exceeds it by > 2^1
constexpr float TAU_S = 2.0f;                // ... and the scale reference if a scale exceeds it 2x
constexpr float P_TOP = 64.0f;
// A head's running max also moves down, to a tile's max that lies more than
// 2^DOWN below it (and within 2^DOWN_CAP of the highest max so far): the weights
// of a bulk of tokens far below an earlier dominant token then stay inside the
// e4m3 range instead of flushing to zero in both terms.
constexpr float DOWN = 10.0f;
constexpr float DOWN_CAP = 60.0f;
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on any single wait

constexpr int align1k(int x) { return (x + 1023) & ~1023; }

// Per head-group width N: ring sizes, barriers, TMEM columns and shared memory.
template <int N>
struct Cfg {
  static constexpr int NB = 2 * N;           // B-operand rows / MMA N: hi terms, then lo terms
  static constexpr int NH = N / 2;           // heads per softmax group
  // ring slots: the Lc blocks (freed by the context MMAs), the Rc blocks (freed
  // by the score MMAs); a block of tile i reuses a slot of tile i - 3 at the
  // oldest while RL <= 12, which keeps the NTF tile barriers exact
  static constexpr int RL = N <= 16 ? 11 : 9;
  static constexpr int RR = 2;
  static_assert(RL >= 5 && RL <= 12, "Lc ring size");
  // barriers
  static constexpr int B_TFULL = 0;                  // [NTF] a tile's scales and blocks loaded
  static constexpr int B_LEMPTY = B_TFULL + NTF;     // [RL] Lc slot read by its context MMAs
  static constexpr int B_REMPTY = B_LEMPTY + RL;     // [RR] Rc slot read by its score MMAs
  static constexpr int B_SFULL = B_REMPTY + RR;      // [2] S of a tile in TMEM
  static constexpr int B_SEMPTY = B_SFULL + 2;       // [2] S read by the softmax (8 arrivals)
  static constexpr int B_PFULL = B_SEMPTY + 2;       // [2] P'' written, O rescaled (8 arrivals)
  static constexpr int B_ODONE = B_PFULL + 2;        // [2] context MMAs of a tile done
  static constexpr int B_G = B_ODONE + 2;            // [2] a softmax group's warps meet (4 arrivals)
  static constexpr int B_DRAIN = B_G + 2;            // [2] the issuers' final drains
  static constexpr int B_QREADY = B_DRAIN + 2;       // the next segment's query is in place (8 arrivals)
  static constexpr int NBAR = B_QREADY + 1;
  // TMEM columns: two S buffers of [S_L hi | S_L lo | S_R hi | S_R lo] (N each),
  // then O: four d-blocks of [hi | lo] (N each)
  static constexpr int S_COLS = 4 * N;
  static constexpr int T_O = 2 * S_COLS;
  static constexpr int TMEM_COLS = 16 * N;
  // shared memory (offsets from the 1024-aligned base)
  static constexpr int OFF_BAR = 0;
  static constexpr int OFF_FLAGS = 256;              // tmem base, abort flag
  static constexpr int OFF_FACTS = 272;              // [NTF] page facts of the tiles in flight
  static constexpr int OFF_RS = 288;                 // [2][2][4] warp maxima of sLc
  static constexpr int OFF_CS = 384;                 // [N] c_h
  static constexpr int OFF_LS = 512;                 // [4][N] denominators per warp
  static constexpr int OFF_RMAX = 1024;              // [2][4][N] warp tile maxima per head
  static constexpr int OFF_SCR = 2048;               // [NTF][128 tokens][2] f32 row scales
  static constexpr int OFF_PT = OFF_SCR + NTF * TILE * 8;  // [PT_PAGES] block-table entries
  // the query: [4 Lc K-blocks][NB rows x 128 B] (128-byte swizzle), then the Rc
  // K-block [NB rows x 64 B] (64-byte swizzle)
  static constexpr int OFF_Q = align1k(OFF_PT + PT_PAGES * 4);
  static constexpr int OFF_P = OFF_Q + 4 * NB * 128 + NB * 64;  // [2][NB rows x 128 tokens]
  static constexpr int OFF_LRING = align1k(OFF_P + 2 * NB * 128);
  static constexpr int OFF_RRING = OFF_LRING + RL * KBLK;
  static constexpr int TOTAL = OFF_RRING + RR * RBLK;
  static constexpr int SMEM = TOTAL + 1024;          // slack for the 1024-byte alignment
  static_assert(NBAR * 8 <= OFF_FLAGS && OFF_FACTS + NTF * 4 <= OFF_RS, "barriers and flags");
  static_assert(OFF_RS + 64 <= OFF_CS && OFF_CS + N * 4 <= OFF_LS, "scratch");
  static_assert(OFF_LS + 4 * N * 4 <= OFF_RMAX && OFF_RMAX + 8 * N * 4 <= OFF_SCR, "scratch");
  static_assert(SMEM <= 232448, "shared memory above the per-CTA limit");
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation");
  static_assert(OFF_P % 1024 == 0 && (OFF_Q + 4 * NB * 128) % 512 == 0, "operand alignment");
};

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

// Byte offset of 16-byte unit u (0..3) of row r in a 64-byte-swizzled K-major
// atom (8 rows of 64 bytes; the unit index turned by bits 1..2 of the row).
__device__ __forceinline__ uint32_t sw64(int r, int u) {
  return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void sts8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <int N>
__global__ void __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap rmap, const __grid_constant__ CUtensorMap smap) {
  using C = Cfg<N>;
  constexpr int NB = C::NB, NH = C::NH, RL = C::RL, RR = C::RR;
  constexpr int LOG2_NH = NH == 8 ? 3 : 4;
  static_assert(NH == 8 || NH == 16, "head groups of 16 or 32");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's work: one or two segments (a range that runs from one (sequence,
  // head group) pair into the next), or one per-sequence item.
  __shared__ Range s_rg;
  if (warp == 0) {
    Range rg;
    if (!find_range(a, blockIdx.x, rg)) {
      WorkItem it;
      const bool ok = find_item(a, blockIdx.x, it);
      rg.n = ok ? 1 : 0;
      if (ok) {
        Segment& sg = rg.s[0];
        sg.b = it.b;
        sg.g = it.g;
        sg.t0 = it.t0;
        sg.t1 = it.t1;
        sg.sid = blockIdx.x;
        sg.first = it.first;
        sg.count = it.count;
        sg.starts = (int64_t)blockIdx.x == it.first;
      }
    }
    if (lane == 0) {
      for (int j = 0; j < rg.n; ++j) record_range_segment(a, rg.s[j]);
      s_rg = rg;
    }
  }
  __syncthreads();
  const int nseg = s_rg.n;
  if (nseg == 0) return;  // past the last work item of this call
  auto seg_tiles = [&](int j) -> int {
    return (int)((s_rg.s[j].t1 - s_rg.s[j].t0 + TILE - 1) / TILE);
  };

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_FLAGS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_FLAGS + 4);
  volatile uint32_t* facts = reinterpret_cast<volatile uint32_t*>(sm + C::OFF_FACTS);
  float* cs = reinterpret_cast<float*>(sm + C::OFF_CS);
  int32_t* pt = reinterpret_cast<int32_t*>(sm + C::OFF_PT);
  const uint32_t scr = smem_u32(sm + C::OFF_SCR);
  const uint32_t qb = smem_u32(sm + C::OFF_Q);
  const uint32_t pb = smem_u32(sm + C::OFF_P);
  const uint32_t lring = smem_u32(sm + C::OFF_LRING);
  const uint32_t rring = smem_u32(sm + C::OFF_RRING);
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(a.err, ERR_TIMEOUT);
  };


  // The query of segment j's heads in the score MMA's B form, by threads tid of
  // nt (the softmax warps, for the first segment and for the second alike):
  // K-block k (Lc channels 128k.., k = 4: Rc) holds NB rows, row h the hi term of
  // head h and row N + h its lo term (rows of 128 bytes, 128-byte swizzle; the Rc
  // block rows of 64 bytes, 64-byte swizzle), and c_h.  Heads past H get zeros and
  // c_h = 0.
  auto load_query = [&](int j, int tid, int nt) {
    const int b = s_rg.s[j].b, h0 = s_rg.s[j].g * N;
    constexpr int QU = 8;  // 16-byte units in flight per thread
    for (int k0 = tid; k0 < N * 72; k0 += QU * nt) {
      uint4 vv[QU];
#pragma unroll
      for (int e = 0; e < QU; ++e) {
        const int k = k0 + e * nt, hh = k / 72, u = k % 72;
        vv[e] = make_uint4(0u, 0u, 0u, 0u);
        if (k < N * 72 && h0 + hh < a.H)
          vv[e] = __ldg(reinterpret_cast<const uint4*>(a.q8 + ((int64_t)b * a.H + h0 + hh) * Q8_BYTES) + u);
      }
#pragma unroll
      for (int e = 0; e < QU; ++e) {
      const int k = k0 + e * nt, hh = k / 72, u = k % 72;
      if (k >= N * 72) break;
      const uint4 v = vv[e];
      int blk, r, uu;
      if (u < 32) {
        blk = u >> 3; uu = u & 7; r = hh;
      } else if (u < 64) {
        blk = (u - 32) >> 3; uu = (u - 32) & 7; r = N + hh;
      } else if (u < 68) {
        blk = 4; uu = u - 64; r = hh;
      } else {
        blk = 4; uu = u - 68; r = N + hh;
      }
      sts128(qb + blk * NB * 128 + (blk < 4 ? sw128(r, uu) : sw64(r, uu)), v);
      }
    }
    for (int st = tid; st < N; st += nt)
      cs[st] = (h0 + st < a.H) ? __ldg(&a.cq[(int64_t)b * a.H + h0 + st]) : 0.f;
    fence_proxy_async_smem();
  };

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < NTF; ++i) mbar_init(&bars[C::B_TFULL + i], 1);
    for (int i = 0; i < RL; ++i) mbar_init(&bars[C::B_LEMPTY + i], 1);
    for (int i = 0; i < RR; ++i) mbar_init(&bars[C::B_REMPTY + i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[C::B_SFULL + i], 1);
      mbar_init(&bars[C::B_SEMPTY + i], NSOFT);
      mbar_init(&bars[C::B_PFULL + i], NSOFT);
      mbar_init(&bars[C::B_ODONE + i], 1);
      mbar_init(&bars[C::B_G + i], NSOFT / 2);
      mbar_init(&bars[C::B_DRAIN + i], 1);
    }
    mbar_init(&bars[C::B_QREADY], NSOFT);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == W_TMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
    load_page_table(a, s_rg.s[0].b, s_rg.s[0].t0, s_rg.s[0].t1, pt, lane);
  } else if (warp >= W_SOFT) {
    grid_dependency_wait();  // the query-prep launch has completed
    load_query(0, threadIdx.x - W_SOFT * 32, NSOFT * 32);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_TMA) {
    // ---------------------------------------------------------- TMA loads
    // Per tile: the row scales (one 128-float box per page), then the Rc block
    // and Lc blocks 0..3, each page a 64-row box; all complete on the tile's
    // barrier, armed once with the tile's bytes.  A block's slot is free once the
    // MMAs that last read it are done.  Tiles are counted across segments (gi),
    // for the rings and the barriers' phases.  The whole warp walks the loop and
    // waits; one elected lane issues.
    bool ok = true;
    int n_req = 0;  // tiles whose barrier has been armed
    int gi = 0;
    for (int j = 0; ok && j < nseg; ++j) {
      const int b = s_rg.s[j].b;
      const int64_t t0 = s_rg.s[j].t0, t_end = s_rg.s[j].t1;
      const int n_tiles = seg_tiles(j);
      if (j > 0) load_page_table(a, b, t0, t_end, pt, lane);
      for (int i = 0; i < n_tiles; ++i, ++gi) {
        const TileRows tr = tile_rows(a, b, t0, t_end, i, pt);
        const uint32_t pages = (tr.s0 >= 0 ? 1u : 0u) + (tr.s1 >= 0 ? 1u : 0u);
        const int tf = gi % NTF, rs = gi % RR;
        uint64_t* tb = &bars[C::B_TFULL + tf];
        if (!mbar_wait_warp(&bars[C::B_REMPTY + rs], ((gi / RR) & 1) ^ 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          const int jb = 4 * gi + blk, ls = jb % RL;
          if (!mbar_wait_warp(&bars[C::B_LEMPTY + ls], ((jb / RL) & 1) ^ 1, abort_flag, WAIT_NS)) {
            ok = false;
            break;
          }
          if (blk == 0) {
            // the tile's page facts travel with its loads (the arrive releases them;
            // every lane stores the same word, the elected one among them)
            facts[tf] = pack_facts(tr);
            mbar_arrive_expect_tx_warp(tb, pages * (2u * PAGE * 4u + 4u * PAGE * 128u + PAGE * 64u));
            n_req = gi + 1;
            const uint32_t sd = scr + tf * TILE * 8, rd = rring + rs * RBLK;
            if (tr.s0 >= 0) {
              tma_load_1d_warp(sd, &smap, (int)(2 * tr.s0), tb);
              tma_load_2d_warp(rd, &rmap, DL, (int)tr.s0, tb);
            }
            if (tr.s1 >= 0) {
              tma_load_1d_warp(sd + 2 * PAGE * 4, &smap, (int)(2 * tr.s1), tb);
              tma_load_2d_warp(rd + PAGE * 64, &rmap, DL, (int)tr.s1, tb);
            }
          }
          const uint32_t ld = lring + ls * KBLK;
          if (tr.s0 >= 0) tma_load_2d_warp(ld, &kmap, 128 * blk, (int)tr.s0, tb);
          if (tr.s1 >= 0) tma_load_2d_warp(ld + PAGE * 128, &kmap, 128 * blk, (int)tr.s1, tb);
        }
        if (!ok) break;
      }
    }
    if (!ok) {
      // after an abort, let the loads already requested land before the CTA can
      // leave (a tile requested in part never completes its barrier: that wait
      // then ends at its bound, after those loads have landed)
      if (lane == 0) fail();
      const int zero = 0;
      for (int i = (n_req > NTF ? n_req - NTF : 0); i < n_req; ++i)
        (void)mbar_wait(&bars[C::B_TFULL + i % NTF], (i / NTF) & 1, &zero, WAIT_NS);
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ---------------------------------------------------------- score MMAs
    // S[t][h] for the NB query rows: A = the tile's block (K-major, 32 bytes of
    // channels per MMA), B = the query's block.  The whole warp walks the loop;
    // one elected lane issues.
    const uint32_t idS = idesc_f16(128, NB, false, false);  // e4m3 x e4m3 (format 0)
    const int split = seg_tiles(0), n_all = split + (nseg > 1 ? seg_tiles(1) : 0);
    bool ok = true;
    for (int i = 0; ok && i < n_all; ++i) {  // tiles counted across segments
      // the second segment's query: the softmax warps put it in place once they
      // have read the first segment's last scores, before that segment's epilogue
      if (i == split && !mbar_wait_warp(&bars[C::B_QREADY], 0, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      const int buf = i & 1;
      if (!mbar_wait_warp(&bars[C::B_SEMPTY + buf], ((i >> 1) & 1) ^ 1, abort_flag, WAIT_NS) ||
          !mbar_wait_warp(&bars[C::B_TFULL + i % NTF], (i / NTF) & 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dL = tmem + buf * C::S_COLS, dR = dL + NB;
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const uint64_t ad = smem_desc(lring + ((4 * i + blk) % RL) * KBLK, 16, 1024, SW128);
        const uint64_t bd = smem_desc(qb + blk * NB * 128, 16, 1024, SW128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f8_warp(dL, ad + 2 * kk, bd + 2 * kk, idS, (blk | kk) != 0);
      }
      {
        const uint64_t ad = smem_desc(rring + (i % RR) * RBLK, 16, 512, SW64);
        const uint64_t bd = smem_desc(qb + 4 * NB * 128, 16, 512, SW64);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) mma_f8_warp(dR, ad + 2 * kk, bd + 2 * kk, idS, kk != 0);
      }
      mma_commit_warp(&bars[C::B_REMPTY + i % RR]);
      mma_commit_warp(&bars[C::B_SFULL + buf]);
    }
    if (!ok && lane == 0) fail();
    // drain: every MMA issued above completes before TMEM is released (this wait
    // ignores the abort flag; it is still bounded in time)
    const int zero = 0;
    mma_commit_warp(&bars[C::B_DRAIN]);
    (void)mbar_wait(&bars[C::B_DRAIN], 0, &zero, WAIT_NS);
    __syncwarp();
  } else if (warp == W_CTX) {
    // ---------------------------------------------------------- context MMAs
    // O[d][h] += V^T P''^T per d-block: A = the Lc block read MN-major (128
    // channels = one swizzle atom; 8-token groups 1 KB apart, 32 tokens per MMA),
    // B = P'' (K-major, NB rows: hi terms then lo terms).  Rows with no data are
    // zeroed first (the score MMAs of the tile are done by then: its P'' follows
    // its S).  The whole warp walks the loop; one elected lane issues.
    const uint32_t idV = idesc_f16(128, NB, true, false);  // e4m3 (format 0), A MN-major
    const int split = seg_tiles(0), n_all = split + (nseg > 1 ? seg_tiles(1) : 0);
    bool ok = true;
    for (int i = 0; ok && i < n_all; ++i) {  // tiles counted across segments
      const bool first = (i == 0 || i == split);  // a segment's first tile starts its O
      const int buf = i & 1;
      if (!mbar_wait_warp(&bars[C::B_PFULL + buf], (i >> 1) & 1, abort_flag, WAIT_NS) ||
          !mbar_wait_warp(&bars[C::B_TFULL + i % NTF], (i / NTF) & 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      const uint32_t f = facts[i % NTF];
      if (f != FULL_TILE) {
        // rows past the item's end, or in a page the block table does not map
        for (int m = 0; m < 4; ++m) {
          const uint32_t vb = lring + ((4 * i + m) % RL) * KBLK;
          for (int u = lane; u < TILE * 8; u += 32)
            if (!row_has(f, u >> 3)) sts128(vb + u * 16, make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      const uint32_t bp = pb + buf * NB * 128;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int ls = (4 * i + m) % RL;
        const uint32_t vb = lring + ls * KBLK;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_warp(tmem + C::T_O + m * NB, smem_desc(vb + kk * 4096, KBLK, 1024, SW128),
                      smem_desc(bp + kk * 32, 16, 1024, SW128), idV, (!first || kk > 0) ? 1u : 0u);
        mma_commit_warp(&bars[C::B_LEMPTY + ls]);
      }
      mma_commit_warp(&bars[C::B_ODONE + buf]);
    }
    if (!ok && lane == 0) fail();
    const int zero = 0;
    mma_commit_warp(&bars[C::B_DRAIN + 1]);
    (void)mbar_wait(&bars[C::B_DRAIN + 1], 0, &zero, WAIT_NS);
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax
    const int sw = warp - W_SOFT;
    const int grp = sw >> 2;                      // head group: heads [grp*NH, grp*NH + NH)
    const int wq = sw & 3;                        // warp within the group
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;          // token row of the tile = TMEM lane
    const int hb = grp * NH;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    float* rmax = reinterpret_cast<float*>(sm + C::OFF_RMAX);  // [2][4][N]
    float* rsm = reinterpret_cast<float*>(sm + C::OFF_RS);     // [2][2][4]
    float* lsum = reinterpret_cast<float*>(sm + C::OFF_LS);    // [4][N]
    // Per head of the group, the same in every thread of the group: the score
    // constant, the running max in use and the highest one so far.  Per thread:
    // the running denominator of its token rows.
    float c[NH], mu[NH], mhi[NH], lp[NH];
    float sref = 0.f;
    int gph = 0;
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_G + grp]);
      return mbar_wait_warp(&bars[C::B_G + grp], (gph++) & 1, abort_flag, WAIT_NS);
    };
    auto tmem_ld_nh = [&](uint32_t addr, uint32_t (&r)[NH]) {
      if constexpr (NH == 16) {
        tmem_ld16(addr, r);
      } else {
        tmem_ld8(addr, r);
      }
    };
    // byte of P''[h][t] in a K-major [NB rows x 128 tokens] block (128-byte
    // swizzle): row h, 16-byte unit t >> 4, byte t & 15
    auto p_off = [&](int h) -> uint32_t {
      return (uint32_t)((h >> 3) * 1024 + (h & 7) * 128 + (((row >> 4) ^ (h & 7)) << 4) + (row & 15));
    };
    bool ok = true;
    int gi = 0;  // tiles counted across segments (rings, buffers, barrier phases)
    for (int seg = 0; ok && seg < nseg; ++seg) {
    const int n_tiles = seg_tiles(seg);
    const int h0 = s_rg.s[seg].g * N;
    if (seg > 0) {
      // every softmax warp has put its share of the query and c_h in place
      if (!mbar_wait_warp(&bars[C::B_QREADY], 0, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      c[h] = cs[hb + h];
      mu[h] = -INFINITY;
      mhi[h] = -INFINITY;
      lp[h] = 0.f;
    }
    sref = 0.f;
    if (seg + 1 < nseg && sw == 0) {
      // the next segment's prepared query (contiguous in global memory) into L2
      // now, so that loading it at the switch does not wait on DRAM
      const Segment& nx = s_rg.s[seg + 1];
      const int64_t q0 = (int64_t)nx.b * a.H + (int64_t)nx.g * N;
      const int64_t nq = (a.H - nx.g * N) < N ? (a.H - nx.g * N) : N;
      prefetch_l2_warp(a.q8 + q0 * Q8_BYTES, (uint32_t)(nq * Q8_BYTES));
    }
    for (int i = 0; i < n_tiles; ++i, ++gi) {
      const int buf = gi & 1, tf = gi % NTF;
      if (!mbar_wait_warp(&bars[C::B_TFULL + tf], (gi / NTF) & 1, abort_flag, WAIT_NS) ||
          !mbar_wait_warp(&bars[C::B_SFULL + buf], (gi >> 1) & 1, abort_flag, WAIT_NS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool valid = row_has(facts[tf], row);
      const float2 s2 = *reinterpret_cast<const float2*>(sm + C::OFF_SCR + (tf * TILE + row) * 8);
      // u = sLc (S_L hi + S_L lo) + sRc (S_R hi + S_R lo); the score in log2 units
      // is z = c_h u with c_h >= 0, so the tile max is taken on u
      float u[NH];
      {
        uint32_t r0[NH], r1[NH], r2[NH], r3[NH];
        const uint32_t sb = tmem + lane_addr + buf * C::S_COLS + hb;
        tmem_ld_nh(sb, r0);
        tmem_ld_nh(sb + N, r1);
        tmem_ld_nh(sb + 2 * N, r2);
        tmem_ld_nh(sb + 3 * N, r3);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float sl = __uint_as_float(r0[h]) + __uint_as_float(r1[h]);
          const float sr = __uint_as_float(r2[h]) + __uint_as_float(r3[h]);
          u[h] = valid ? fmaf(s2.y, sr, s2.x * sl) : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_SEMPTY + buf]);

      // tile maxima per head and of sLc over the group's four warps
      {
        const float mx = warp_transpose_reduce<NH, true>(u, lane);
        if ((lane & ((32 >> LOG2_NH) - 1)) == 0)
          rmax[(buf * 4 + wq) * N + hb + (lane >> (5 - LOG2_NH))] = mx;
        float smax = valid ? s2.x : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) rsm[(buf * 2 + grp) * 4 + wq] = smax;
      }
      if (!group_sync()) {
        ok = false;
        break;
      }
      // Lazy maxima, worked out by every thread of the group from the same
      // values: a head's max moves up when the tile's exceeds it by more than
      // 2^TAU, down when the tile's lies more than 2^DOWN below it (and within
      // 2^DOWN_CAP of the highest so far); the scale reference moves when a scale
      // exceeds it TAU_S times.  fc = the factor of the head's O columns.
      float al[NH], fc[NH];
      bool corr = false;
      {
        const float* rm = rmax + buf * 4 * N + hb;
        const float* rq = rsm + (buf * 2 + grp) * 4;
        const float gmax = fmaxf(fmaxf(rq[0], rq[1]), fmaxf(rq[2], rq[3]));
        const float sref_new = (gmax > sref * TAU_S) ? gmax : sref;
        const float beta = (sref_new == sref) ? 1.f : (sref > 0.f ? sref / sref_new : 0.f);
        sref = sref_new;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float umax = fmaxf(fmaxf(rm[h], rm[N + h]), fmaxf(rm[2 * N + h], rm[3 * N + h]));
          const float tmax = c[h] > 0.f ? c[h] * umax : -INFINITY;
          float mn = mu[h];
          if (tmax > mu[h] + TAU) {
            mn = tmax;
          } else if (tmax < mu[h] - DOWN && tmax >= mhi[h] - DOWN_CAP && tmax > -INFINITY) {
            mn = tmax;
          }
          al[h] = 1.f;
          if (mn != mu[h]) {
            al[h] = (mu[h] == -INFINITY) ? 0.f : ex2_approx(mu[h] - mn);
            mu[h] = mn;
          }
          mhi[h] = fmaxf(mhi[h], mu[h]);
          fc[h] = al[h] * beta;
          corr |= (fc[h] != 1.f);
        }
        corr = corr && i > 0;  // tile 0's MMAs initialise O
      }

      // p = 2^(z - m) (0 for rows without data and for heads past H), the running
      // denominators, and P'' = p sLc P_TOP / s_ref as e4m3 hi + lo, computed in
      // f16 (the residual of the hi term is exact there); bytes packed by head
      const float w = valid ? s2.x * (sref > 0.f ? P_TOP / sref : 0.f) : 0.f;
      uint32_t phi[NH / 4], plo[NH / 4];
#pragma unroll
      for (int h = 0; h < NH; h += 4) {
        float z[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int hh = h + j;
          const float mneg = c[hh] > 0.f ? -fmaxf(mu[hh], -3.0e38f) : -INFINITY;
          const float p = valid ? ex2_approx(fmaf(c[hh], u[hh], mneg)) : 0.f;
          lp[hh] = fmaf(lp[hh], al[hh], p);
          z[j] = p * w;
        }
        const __half2 x01 = __floats2half2_rn(z[0], z[1]);
        const __half2 x23 = __floats2half2_rn(z[2], z[3]);
        const uint16_t h01 = f16x2_to_e4m3x2(x01), h23 = f16x2_to_e4m3x2(x23);
        const uint32_t d01 = e4m3x2_to_f16x2(h01), d23 = e4m3x2_to_f16x2(h23);
        const uint16_t l01 = f16x2_to_e4m3x2(__hsub2(x01, *reinterpret_cast<const __half2*>(&d01)));
        const uint16_t l23 = f16x2_to_e4m3x2(__hsub2(x23, *reinterpret_cast<const __half2*>(&d23)));
        phi[h / 4] = (uint32_t)h01 | ((uint32_t)h23 << 16);
        plo[h / 4] = (uint32_t)l01 | ((uint32_t)l23 << 16);
      }
      if (corr) {
        // O columns may change only once the previous tile's context MMAs are done
        if (!mbar_wait_warp(&bars[C::B_ODONE + (buf ^ 1)], ((gi - 1) >> 1) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // rescale the hi and lo columns of the heads whose factor moved, 8 heads at
        // a time, the four d-blocks' loads in flight together
#pragma unroll
        for (int c8 = 0; c8 < NH; c8 += 8) {
          bool moved = false;
#pragma unroll
          for (int j = 0; j < 8; ++j) moved |= (fc[c8 + j] != 1.f);
          if (!moved) continue;  // the same in every thread of the group
#pragma unroll 1
          for (int term = 0; term < 2; ++term) {
            uint32_t r[4][8];
#pragma unroll
            for (int m = 0; m < 4; ++m)
              tmem_ld8(tmem + lane_addr + C::T_O + m * NB + term * N + hb + c8, r[m]);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int j = 0; j < 8; ++j) r[m][j] = __float_as_uint(__uint_as_float(r[m][j]) * fc[c8 + j]);
              tmem_st8(tmem + lane_addr + C::T_O + m * NB + term * N + hb + c8, r[m]);
            }
          }
        }
        tmem_wait_st();
      } else if (gi >= 2) {
        // the P'' buffer is free once the context MMAs of tile gi - 2 are done
        if (!mbar_wait_warp(&bars[C::B_ODONE + buf], ((gi >> 1) & 1) ^ 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
      }
      const uint32_t pbb = pb + buf * NB * 128;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        sts8(pbb + p_off(hb + h), phi[h / 4] >> (8 * (h & 3)));
        sts8(pbb + p_off(N + hb + h), plo[h / 4] >> (8 * (h & 3)));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_PFULL + buf]);
    }
    if (!ok) break;
    if (seg + 1 < nseg) {
      // the next segment's query: this warp has seen this segment's last scores,
      // so the score MMAs that read the query are done; the next segment's first
      // scores then overlap this segment's last context MMAs and epilogue
      load_query(seg + 1, threadIdx.x - W_SOFT * 32, NSOFT * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_QREADY]);
    }
    {
      ok = mbar_wait_warp(&bars[C::B_ODONE + ((gi - 1) & 1)], ((gi - 1) >> 1) & 1,
                          abort_flag, WAIT_NS);
      if (ok) {
        // denominators: the per-thread partials of each head over the 128 rows
        const float ls = warp_transpose_reduce<NH, false>(lp, lane);
        if ((lane & ((32 >> LOG2_NH) - 1)) == 0) lsum[wq * N + hb + (lane >> (5 - LOG2_NH))] = ls;
        ok = group_sync();
      }
      if (ok) {
        tc_fence_after();
        const int64_t base = s_rg.s[seg].sid * N;  // this segment's partials
        if (wq == 0 && lane < NH && h0 + hb + lane < a.H) {
          float m_h = mu[0];
#pragma unroll
          for (int h = 1; h < NH; ++h) m_h = (lane == h) ? mu[h] : m_h;
          const int hh = hb + lane;
          a.ws_m[base + hh] = m_h;
          a.ws_l[base + hh] = (lsum[hh] + lsum[N + hh]) + (lsum[2 * N + hh] + lsum[3 * N + hh]);
        }
        // unnormalised partial o = (O hi + O lo) s_ref / P_TOP
        const float oscale = sref * (1.0f / P_TOP);
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int c8 = 0; c8 < NH; c8 += 8) {
            uint32_t rh[8], rl[8];
            tmem_ld8(tmem + lane_addr + C::T_O + m * NB + hb + c8, rh);
            tmem_ld8(tmem + lane_addr + C::T_O + m * NB + N + hb + c8, rl);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int h = hb + c8 + j;
              if (h0 + h < a.H)
                a.ws_o[(base + h) * DL + m * 128 + row] =
                    (__uint_as_float(rh[j]) + __uint_as_float(rl[j])) * oscale;
            }
          }
        }
      }
    }
    }  // segments
    if (!ok && lane == 0) fail();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_TMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int N>
cudaError_t launch_n(const DecodeArgs& a, cudaStream_t s) {
  static std::atomic<int> memo[MAX_DEVICES];
  int done = 0;
  cudaError_t e = per_device(memo, [](int* v) {
    *v = 1;
    return cudaFuncSetAttribute(decode_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<N>::SMEM);
  }, &done);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap, rmap, smap;
  e = make_cache_map(a, &kmap);
  if (e != cudaSuccess) return e;
  e = make_rc_map(a, &rmap);
  if (e != cudaSuccess) return e;
  e = make_scale_map(a, &smap);
  if (e != cudaSuccess) return e;
  e = launch_prep_query(a, s);
  if (e != cudaSuccess) return e;
  return launch_after_prep(decode_tc_kernel<N>, a.plan.max_items, NTHREADS, Cfg<N>::SMEM, s, a, kmap,
                           rmap, smap);
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

// Tensor map of the cache's Rc bytes (columns 512..575): boxes of 64 rows x 64
// bytes, 64-byte swizzle, for the one-CTA kernel's 8 KB Rc slots.
cudaError_t make_rc_map(const DecodeArgs& a, CUtensorMap* map) {
  const int64_t rows = a.block_table != nullptr ? a.n_blocks * PAGE : a.T_contig;
  if (rows < 1 || a.codes == nullptr) {
    memset(map, 0, sizeof(*map));
    return cudaSuccess;
  }
  if (rows >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D};
  const cuuint32_t box[2] = {64, PAGE};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.codes), dims,
                      strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// 1-D tensor map of the row scales (f32, two per slot): boxes of 128 floats (one
// page); floats past the end read as zeros.
cudaError_t make_scale_map(const DecodeArgs& a, CUtensorMap* map) {
  const int64_t rows = a.block_table != nullptr ? a.n_blocks * PAGE : a.T_contig;
  if (rows < 1 || a.scales == nullptr) {
    memset(map, 0, sizeof(*map));
    return cudaSuccess;
  }
  if (2 * rows >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  const cuuint64_t dims[1] = {(cuuint64_t)(2 * rows)};
  const cuuint64_t strides[1] = {(cuuint64_t)(2 * rows) * 4};  // unused for one dimension
  const cuuint32_t box[1] = {2 * PAGE};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(a.scales), dims,
                      strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool tc_available() { return true; }

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  switch (a.plan.hg) {
    case 16: return launch_n<16>(a, s);
    case 32: return launch_n<32>(a, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kv8
