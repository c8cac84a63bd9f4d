// decode_pair.cu -- split-T absorbed MLA decode on pairs of SMs (a cluster of
// two CTAs) for groups of 128 heads: one CTA computes the scores and the
// softmax, the other the context, both on tcgen05 tensor cores with e4m3
// operands and f32 accumulators in TMEM.
//
// Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description: the latent Lc is both key and value of the
// absorbed attention, the RoPE part Rc is key only, and each row's f32 scale is
// applied outside its dot product; closing note: split-T kernels for long
// caches.  Per (sequence b, head h):
//   z_t = sm * ( sLc_t <q_lat, dec(Lc_t)> + sRc_t <q_rope, dec(Rc_t)> )
//   o   = sum_t softmax(z)_t sLc_t dec(Lc_t)
//
// A work item is (sequence, group of 128 heads, range of 128-token tiles); a
// cluster of two CTAs takes one item.
//
// Score CTA (rank 0), per tile:
//   S[h][t] = Q_h . K_t   kind::f8f6f4, M = 128 heads, N = 128 tokens, K = 512
//             (S_L) and 64 (S_R) in two TMEM accumulators (the row scales of Lc
//             and Rc differ).  A = the query in two e4m3 terms (hi + the e4m3
//             residual) on one per-head power-of-two scale: its Lc part in TMEM,
//             its Rc part in shared memory.  B = the e4m3 cache tile itself,
//             loaded by TMA (five [128 tokens x 128 bytes] blocks: Lc 0..3 and Rc,
//             whose box runs past column 576 into zero fill), never converted.
//   softmax   sixteen warps, four per TMEM lane quarter; a thread owns one head
//             (its TMEM lane) and one part (32 tokens) of the tile: z = c_h (sLc
//             S_L + sRc S_R), tile maximum per head over the four parts, lazy
//             running maxima, running denominators of the exact weights
//             p = 2^(z - m_h), and p as f16.  Each warp stages its 32 heads x 32
//             tokens of p, its heads' O rescale factors and its part's token
//             weights w_t = sLc_t P_TOP / s_ref in shared memory and sends them
//             with one bulk copy to the context CTA.
// Context CTA (rank 1), per tile:
//   sixteen warps turn the received p into the context operand in place,
//   P''[h][t] = p w_t (f16) as two e4m3 terms, hi + lo; zero the V rows without
//   data; rescale the O rows of heads whose factor moved, one half of O while the
//   MMAs of the other half run; and write the partial o at the end (each head's
//   O half-row put in a padded shared-memory row and sent by one bulk copy).
//   O[h][d] += sum_t P''[h][t] V[t][d]   kind::f8f6f4, M = 128 heads, N = 256
//             latent channels (two halves of 512), K = 32 tokens per MMA, hi and
//             lo terms into the same accumulator (all 512 TMEM columns).  V is the
//             e4m3 cache tile (Lc, by TMA), read as an MN-major operand.
// The two MMA-issuing threads wait on as few barriers as possible (one per tile
// for the scores, one per O half for the context): a barrier wait on the issuing
// thread leaves the tensor pipe idle for about two hundred cycles.
//
// Lazy maxima: a head's running maximum moves up when a tile's maximum exceeds
// it by more than 2^TAU, and down to the tile's maximum when that lies more than
// 2^DOWN below it (but within 2^DOWN_CAP of the highest maximum so far), so that
// the weights of a bulk of tokens far below an earlier dominant token stay inside
// the e4m3 range instead of flushing to zero; the row-scale reference moves when a
// scale exceeds it TAU_S times.  Every wait is bounded (2 s): on a timeout the CTA
// flags the workspace error word, drains its MMAs and copies, meets its partner
// at the closing cluster barrier, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {

namespace {

using namespace ptx;

constexpr int HG = 128;                      // heads per work item
constexpr int W_TMA = 0, W_MMA = 1, W_LANE = 2;
constexpr int N_LANE_WARPS = 16;             // four per TMEM lane quarter
constexpr int NTHREADS = (W_LANE + N_LANE_WARPS) * 32;
constexpr int PART = TILE / 4;               // 32 tokens: a lane warp's share of a tile
constexpr int KBLK = TILE * 128;             // 16 KB: [128 tokens x 128 bytes]
constexpr int BLKS = 5;                      // K blocks per tile: Lc 0..3, Rc
constexpr int NKS = 2 * BLKS;                // K-block ring slots (score CTA): two tiles
constexpr int NSC = 4;                       // scale ring slots (score CTA), one tile each
constexpr int VTILE = 4 * KBLK;              // 64 KB: the tile's Lc, four d-blocks
constexpr int NVT = 2;                       // V ring slots (context CTA), one tile each
// Payload of one tile, one chunk per lane warp (chunk c = part * 4 + lane
// quarter; the context CTA registers the bytes it expects on its own barrier):
// p as f16 for its 32 heads x 32 tokens (rows of 64 bytes, 16-byte units
// swizzled by the row), the O rescale factors of its heads, the token weights of
// its part (f16), and s_ref.
constexpr int C_P16 = 0, C_FCOL = 32 * PART * 2, C_W = C_FCOL + 32 * 4, C_EXTRA = C_W + PART * 2;
constexpr int CHUNK = C_EXTRA + 16;          // 2256 bytes
constexpr int P_BYTES = N_LANE_WARPS * CHUNK;
constexpr int P_STRIDE = 37 * 1024;
constexpr int L2_AHEAD = 3;                  // tiles prefetched into L2 ahead of the K loads
constexpr float TAU = 1.0f;
constexpr float TAU_S = 2.0f;
constexpr float P_TOP = 64.0f;               // P'' <= 2^TAU * TAU_S * P_TOP = 256 <= 448
constexpr float DOWN = 10.0f;
constexpr float DOWN_CAP = 60.0f;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;

// mbarriers, indices derived from the ring sizes (the payload-free pair sits at
// the same offset in both CTAs: the context CTA's commit multicasts to it)
constexpr int B_PFREE = 0;                   // [2] score: the context MMAs of the payload buffer's last tile are done
constexpr int B_KT = B_PFREE + 2;            // [2] score: all K blocks of a tile loaded (by tile parity)
constexpr int B_KEMPTY = B_KT + 2;           // [2] score: a tile's K blocks consumed by its score MMAs (by tile parity)
constexpr int B_SCFULL = B_KEMPTY + 2;       // [NSC] score: row scales of a tile loaded
constexpr int B_SFULL = B_SCFULL + NSC;      // score: S of a tile in TMEM
constexpr int B_SEMPTY = B_SFULL + 1;        // score: S read and next tile's K loaded (16 arrivals)
constexpr int B_PX = B_SEMPTY + 1;           // [4] score: the four warps of a lane quarter meet
constexpr int B_VT = B_PX + 4;               // [NVT] context: V tile loaded
constexpr int B_VEMPTY = B_VT + NVT;         // [NVT] context: V tile consumed
constexpr int B_PFULL = B_VEMPTY + NVT;      // [2] context: payload of a tile arrived (bulk-copy bytes)
constexpr int B_CVT = B_PFULL + 2;           // context: the payload is read, its buffer may be overwritten (16 arrivals)
constexpr int B_RS = B_CVT + 1;              // [2] context: operand, V rows and O half ready (16 arrivals)
constexpr int B_ODONE = B_RS + 2;            // [2] context: MMAs of an O half done
constexpr int B_DRAIN = B_ODONE + 2;
constexpr int B_QREADY = B_DRAIN + 1;        // score: the query is in TMEM and shared memory (16 arrivals)
constexpr int NBAR = B_QREADY + 1;

// shared memory (offsets from the 1024-aligned base)
constexpr int OFF_BAR = 0;
constexpr int OFF_FLAGS = 512;               // tmem base, abort flag
constexpr int OFF_FACTS = OFF_FLAGS + 16;    // [4] page facts of the tiles in the scale / V ring
constexpr int OFF_XMAX = 1024;               // score: [2 tiles][4 parts][128] part maxima
constexpr int OFF_XSM = OFF_XMAX + 8 * HG * 4;  // score: [2 tiles][4 parts][4] part row-scale maxima
constexpr int OFF_XL = OFF_XSM + 32 * 4;     // score: [4 parts][128] denominators
constexpr int OFF_QR = 8192;                 // score: [128 heads x 128 bytes]: Rc query hi | lo
constexpr int OFF_KRING = OFF_QR + KBLK;
constexpr int OFF_SCR = OFF_KRING + NKS * KBLK;  // [NSC][128 tokens][2] f32
constexpr int OFF_STG = OFF_SCR + NSC * TILE * 8;  // [16 warps] staged payload chunks
constexpr int TOTAL_S = OFF_STG + P_BYTES;
constexpr int OFF_P = 4096;                  // context: 2 payloads / context operands
constexpr int OFF_VRING = OFF_P + 2 * P_STRIDE;
constexpr int TOTAL_C = OFF_VRING + NVT * VTILE;
constexpr int O_ROW = 64 * 4 + 16;           // context epilogue: one head's 64 columns, padded
constexpr int OFF_PT = TOTAL_S > TOTAL_C ? TOTAL_S : TOTAL_C;  // both CTAs: [PT_PAGES] int32
constexpr int SMEM = OFF_PT + PT_PAGES * 4 + 1024;
// score CTA TMEM columns: S_L, S_R (one tile), then the Lc query's hi and lo terms
// (e4m3, four channels per column) as the A operand of the score MMAs
constexpr int T_SL = 0, T_SR = 128, T_QH = 256, T_QL = 384;
static_assert(OFF_XL + 4 * HG * 4 <= OFF_QR, "score CTA scratch overlaps the Rc query");
static_assert(NBAR * 8 <= OFF_FLAGS && OFF_FACTS + 16 <= OFF_XMAX, "barriers, flags and facts overlap");
static_assert(P_BYTES <= P_STRIDE && (P_STRIDE % 1024) == 0 && (OFF_VRING % 1024) == 0,
              "payload layout");
static_assert(2 * KBLK <= P_BYTES, "the context operand (hi and lo atoms) fits in its payload buffer");
static_assert(OFF_P + N_LANE_WARPS * 32 * O_ROW <= TOTAL_C, "the epilogue's staging fits in the payloads and V ring");
static_assert((CHUNK % 16) == 0 && (OFF_STG % 16) == 0, "bulk-copied chunks");
static_assert(SMEM <= 232448, "shared memory above the per-CTA limit");

// byte offset of 16-byte unit u (0..3) of head row r of a payload chunk: rows of
// 64 bytes, the unit index turned by the row so that the eight rows a quarter
// warp touches at once fall on distinct banks
__device__ __forceinline__ uint32_t prow(int r, int u) {
  return (uint32_t)(r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}

// Two e4m3 terms of four f32 values already on the head's scale: hi = e4m3(x),
// lo = e4m3(x - hi) (the difference is exact in f32).
__device__ __forceinline__ void split4(const float* x, uint32_t& hi, uint32_t& lo) {
  const uint16_t h01 = f32x2_to_e4m3x2(x[0], x[1]), h23 = f32x2_to_e4m3x2(x[2], x[3]);
  const uint32_t f01 = e4m3x2_to_f16x2(h01), f23 = e4m3x2_to_f16x2(h23);
  const float2 d01 = __half22float2(*reinterpret_cast<const __half2*>(&f01));
  const float2 d23 = __half22float2(*reinterpret_cast<const __half2*>(&f23));
  const uint16_t l01 = f32x2_to_e4m3x2(x[0] - d01.x, x[1] - d01.y);
  const uint16_t l23 = f32x2_to_e4m3x2(x[2] - d23.x, x[3] - d23.y);
  hi = (uint32_t)h01 | ((uint32_t)h23 << 16);
  lo = (uint32_t)l01 | ((uint32_t)l23 << 16);
}

// Two e4m3 terms of an f16 pair, in f16 arithmetic (the residual of the hi term
// is exact there).
__device__ __forceinline__ void split_h2(__half2 x, uint16_t& hi, uint16_t& lo) {
  hi = f16x2_to_e4m3x2(x);
  const uint32_t d = e4m3x2_to_f16x2(hi);
  lo = f16x2_to_e4m3x2(__hsub2(x, *reinterpret_cast<const __half2*>(&d)));
}

// Packed pairs of f32 (element 0 in the low half) and the sm_100 two-lane f32
// instructions; each lane is rounded exactly as the scalar instruction would be.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// tokens with data in part k (tokens [32 k, 32 k + 32)) of the tile
__device__ __forceinline__ int part_tokens(uint32_t f, int k) {
  const int n = (int)(f & 0xFFu) - PART * k;
  return ((f >> (8 + (k >> 1))) & 1u) ? min(max(n, 0), PART) : 0;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    decode_pair_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap smap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int64_t item = blockIdx.x >> 1;
  __shared__ WorkItem s_it;
  __shared__ int s_ok;
  if (warp == 0) {
    WorkItem it;
    const bool ok = find_item(a, item, it);
    if (lane == 0 && ok && rank == 0) record_segment(a, item, it);
    if (lane == 0) {
      s_it = it;
      s_ok = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;  // past the last work item: both CTAs of the pair leave here
  const int b = s_it.b;
  const int h0 = s_it.g * HG;
  const int64_t t0 = s_it.t0, t_end = s_it.t1;
  const int n_tiles = (int)((t_end - t0 + TILE - 1) / TILE);

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_FLAGS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_FLAGS + 4);
  uint32_t* facts = reinterpret_cast<uint32_t*>(sm + OFF_FACTS);
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(a.err, ERR_TIMEOUT);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_PFREE + i], 1);
      mbar_init(&bars[B_KT + i], 1);
      mbar_init(&bars[B_PFULL + i], 1);
      mbar_init(&bars[B_RS + i], N_LANE_WARPS);
      mbar_init(&bars[B_ODONE + i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&bars[B_KEMPTY + i], 1);
    for (int i = 0; i < NSC; ++i) mbar_init(&bars[B_SCFULL + i], 1);
    mbar_init(&bars[B_SFULL], 1);
    mbar_init(&bars[B_SEMPTY], N_LANE_WARPS);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_PX + i], N_LANE_WARPS / 4);
    for (int i = 0; i < NVT; ++i) {
      mbar_init(&bars[B_VT + i], 1);
      mbar_init(&bars[B_VEMPTY + i], 1);
    }
    mbar_init(&bars[B_CVT], N_LANE_WARPS);
    mbar_init(&bars[B_DRAIN], 1);
    mbar_init(&bars[B_QREADY], N_LANE_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the context CTA expects the payloads of its first two tiles (one per
    // buffer); each later one is expected when its buffer's previous tile is read
    if (rank == 1) {
      mbar_arrive_expect_tx(&bars[B_PFULL], (uint32_t)P_BYTES);
      if (n_tiles > 1) mbar_arrive_expect_tx(&bars[B_PFULL + 1], (uint32_t)P_BYTES);
    }
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();  // the TMEM base address is in shared memory
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised before any remote arrive or copy
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (rank == 0) {
    // ================================================================ score CTA
    const uint32_t kring = smem_u32(sm + OFF_KRING);
    const uint32_t qr = smem_u32(sm + OFF_QR);
    const uint32_t scr = smem_u32(sm + OFF_SCR);
    if (warp == W_TMA) {
      // The whole warp walks the loop and waits; one elected lane issues.
      int32_t* pt = reinterpret_cast<int32_t*>(sm + OFF_PT);
      load_page_table(a, b, t0, t_end, pt, lane);
      bool ok = true;
      auto prefetch_tile = [&](int i) {
        const int64_t tb = t0 + (int64_t)i * TILE;
        for (int pg = 0; pg < 2; ++pg) {
          const int64_t tk = tb + pg * PAGE;
          if (tk >= t_end) break;
          const int64_t nt = (t_end - tk < PAGE) ? t_end - tk : PAGE;
          const int64_t slot = item_slot(a, b, tk, t0, pt);
          if (slot >= 0) prefetch_l2_warp(a.codes + slot * D, (uint32_t)(nt * D));
        }
      };
      int nk = 0, nsc = 0;  // tiles whose K blocks / row scales were requested
      for (int i = 0; ok && i < n_tiles; ++i) {
        const TileRows tr = tile_rows(a, b, t0, t_end, i, pt);
        const uint32_t pages = (tr.s0 >= 0 ? 1u : 0u) + (tr.s1 >= 0 ? 1u : 0u);
        const int sc = i % NSC;
        // the tile's five blocks complete on one barrier and take the slots of the
        // tile two before, free once that tile's score MMAs are done (one wait per
        // tile, then every load at once).  Those MMAs started after the softmax
        // warps had released tile i - 3, and a warp reads every row scale and page
        // fact of a tile before it releases it, so the scale slot of tile i - 4 is
        // free then too.
        uint64_t* kt = &bars[B_KT + (i & 1)];
        if (!mbar_wait_warp(&bars[B_KEMPTY + (i & 1)], ((i >> 1) & 1) ^ 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        // the tile's page facts travel with its row scales (the arrive releases them;
        // every lane stores the same word, the elected one among them)
        facts[sc] = pack_facts(tr);
        mbar_arrive_expect_tx_warp(&bars[B_SCFULL + sc], 512u * pages);
        if (tr.s0 >= 0) tma_load_1d_warp(scr + sc * TILE * 8, &smap, (int)(2 * tr.s0), &bars[B_SCFULL + sc]);
        if (tr.s1 >= 0)
          tma_load_1d_warp(scr + sc * TILE * 8 + 512, &smap, (int)(2 * tr.s1), &bars[B_SCFULL + sc]);
        nsc = i + 1;
        mbar_arrive_expect_tx_warp(kt, 8192u * pages * BLKS);
        nk = i + 1;
#pragma unroll 1
        for (int blk = 0; blk < BLKS; ++blk) {
          const uint32_t dst = kring + ((i & 1) * BLKS + blk) * KBLK;
          if (tr.s0 >= 0) tma_load_2d_warp(dst, &kmap, 128 * blk, (int)tr.s0, kt);
          if (tr.s1 >= 0) tma_load_2d_warp(dst + 8192, &kmap, 128 * blk, (int)tr.s1, kt);
        }
        // then the L2 prefetch of the tiles ahead (the next tile is loaded at once;
        // after the first, the one L2_AHEAD tiles on)
        for (int j = (i == 0 ? 2 : i + L2_AHEAD); ok && j <= i + L2_AHEAD && j < n_tiles; ++j)
          prefetch_tile(j);
      }
      if (!ok) {
        // after an abort, let the loads already requested land before the CTA can
        // leave (a tile requested in part never completes its barrier: the wait
        // then ends at its bound, after those loads have landed)
        if (lane == 0) fail();
        const int zero = 0;
        for (int i = (nk > 2 ? nk - 2 : 0); i < nk; ++i)
          (void)mbar_wait(&bars[B_KT + (i & 1)], (i >> 1) & 1, &zero, WAIT_NS);
        for (int i = (nsc > NSC ? nsc - NSC : 0); i < nsc; ++i)
          (void)mbar_wait(&bars[B_SCFULL + i % NSC], (i / NSC) & 1, &zero, WAIT_NS);
      }
      __syncwarp();
    } else if (warp == W_MMA) {
      // The whole warp walks the loop and waits; one elected lane issues.
      const uint32_t idS = idesc_f16(128, 128, false, false);  // e4m3 x e4m3 (format 0)
      const uint64_t kdesc = smem_desc(kring, 16, 1024, SW128);
      const uint64_t qdesc = smem_desc(qr, 16, 1024, SW128);
      // the query, and tile 0's K blocks; a later tile's are waited for by the
      // softmax warps before they release S, so one barrier per tile gates these MMAs
      bool ok = mbar_wait_warp(&bars[B_QREADY], 0, abort_flag, WAIT_NS) &&
                mbar_wait_warp(&bars[B_KT], 0, abort_flag, WAIT_NS);
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (!mbar_wait_warp(&bars[B_SEMPTY], (i & 1) ^ 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int blk = 0; blk < BLKS; ++blk) {
          const uint64_t bd = kdesc + (uint64_t)((((i & 1) * BLKS + blk) * KBLK) >> 4);
          if (blk < 4) {
            // A = the Lc query from TMEM: 8 columns (32 channels) per MMA
            const uint32_t ah = tmem + T_QH + blk * 32, al = tmem + T_QL + blk * 32;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              mma_f8_ts_warp(tmem + T_SL, ah + kk * 8, bd + 2 * kk, idS, (blk | kk) != 0);
              mma_f8_ts_warp(tmem + T_SL, al + kk * 8, bd + 2 * kk, idS, 1u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              mma_f8_warp(tmem + T_SR, qdesc + 2 * kk, bd + 2 * kk, idS, kk != 0);
              mma_f8_warp(tmem + T_SR, qdesc + 4 + 2 * kk, bd + 2 * kk, idS, 1u);
            }
          }
        }
        mma_commit_warp(&bars[B_KEMPTY + (i & 1)]);
        mma_commit_warp(&bars[B_SFULL]);
      }
      if (!ok && lane == 0) fail();
      const int zero = 0;
      mma_commit_warp(&bars[B_DRAIN]);
      (void)mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
      __syncwarp();
    } else {
      // ---------------------------------------------------------- softmax
      const int q = warp & 3;                  // TMEM lane quarter
      const int part = (warp - W_LANE) >> 2;   // part of the tile: tokens [32 part, 32 part + 32)
      const int hh = q * 32 + lane;            // head of the group = TMEM lane
      const int chunk = part * 4 + q;          // this warp's payload chunk
      const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
      float* xmax = reinterpret_cast<float*>(sm + OFF_XMAX);  // [2][4][128]
      float* xsm = reinterpret_cast<float*>(sm + OFF_XSM);    // [2][4][4]
      float* xl = reinterpret_cast<float*>(sm + OFF_XL);      // [4][128]
      uint8_t* stg_p = sm + OFF_STG + chunk * CHUNK;
      const uint32_t stg = smem_u32(stg_p);
      // The prepared query (two e4m3 terms on the head's power-of-two scale, c_h
      // folding the scale back in with sm_scale * log2(e)): thread (head hh, part)
      // puts Lc channels [128 part, 128 part + 128) of both terms into TMEM lane hh
      // (four channels per column), part 0 also the Rc terms into row hh of the Rc
      // operand in shared memory (hi in bytes 0..63, lo in 64..127).  Heads past H
      // are zeros.  The loads overlap the first tiles' K loads.
      const bool real = h0 + hh < a.H;
      grid_dependency_wait();  // the query-prep launch has completed
      const float c = real ? __ldg(a.cq + (int64_t)b * a.H + h0 + hh) : 0.f;
      {
        const uint4* q8 = reinterpret_cast<const uint4*>(a.q8 + ((int64_t)b * a.H + h0 + hh) * Q8_BYTES);
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {  // 64 channels (16 columns) of each term at a time
          uint32_t hw[16], lw[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int u = 8 * part + 4 * hl + k;
            const uint4 vh = real ? __ldg(q8 + u) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 vl = real ? __ldg(q8 + 32 + u) : make_uint4(0u, 0u, 0u, 0u);
            hw[4 * k] = vh.x; hw[4 * k + 1] = vh.y; hw[4 * k + 2] = vh.z; hw[4 * k + 3] = vh.w;
            lw[4 * k] = vl.x; lw[4 * k + 1] = vl.y; lw[4 * k + 2] = vl.z; lw[4 * k + 3] = vl.w;
          }
          __syncwarp();
          tmem_st16(tmem + lane_addr + T_QH + part * 32 + 16 * hl, hw);
          tmem_st16(tmem + lane_addr + T_QL + part * 32 + 16 * hl, lw);
        }
        if (part == 0) {
          const uint32_t qr = smem_u32(sm + OFF_QR);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            sts128(qr + sw128(hh, u), real ? __ldg(q8 + 64 + u) : make_uint4(0u, 0u, 0u, 0u));
        }
        __syncwarp();
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_QREADY]);
      }
      const bool live = c > 0.f;               // a real head (padding heads have c = 0)
      const uint32_t prem = map_to(smem_u32(sm + OFF_P), 1) + chunk * CHUNK;  // partner's buffers
      const uint32_t pfull_rem = map_to(smem_u32(&bars[B_PFULL]), 1);
      float mu = -INFINITY, mhi = -INFINITY, lsum = 0.f, sref = 0.f;
      int px_phase = 0;
      bool ok = true;
      auto quarter_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_PX + q]);
        return mbar_wait_warp(&bars[B_PX + q], (px_phase++) & 1, abort_flag, WAIT_NS);
      };
      for (int i = 0; i < n_tiles; ++i) {
        const int buf = i & 1, sc = i % NSC, pb = i & 1;
        // the tile's row scales and S, and the next tile's K blocks (waited for here
        // by every warp, so that the MMA thread's one wait per tile covers both)
        if (!mbar_wait_warp(&bars[B_SCFULL + sc], (i / NSC) & 1, abort_flag, WAIT_NS) ||
            !mbar_wait_warp(&bars[B_SFULL], i & 1, abort_flag, WAIT_NS) ||
            (i + 1 < n_tiles &&
             !mbar_wait_warp(&bars[B_KT + ((i + 1) & 1)], ((i + 1) >> 1) & 1, abort_flag, WAIT_NS))) {
          ok = false;
          break;
        }
        const int my_n = part_tokens(facts[sc], part);
        tc_fence_after();
        // S for this thread's head and the part's 32 tokens: both loads in flight at
        // once, and S released as soon as they land (the next tile's score MMAs
        // overwrite it while this tile's softmax runs)
        uint32_t rl[PART], rr[PART];
        tmem_ld32(tmem + lane_addr + T_SL + part * PART, rl);
        tmem_ld32(tmem + lane_addr + T_SR + part * PART, rr);
        // meanwhile: this warp's previous payload copy has read its staging chunk,
        // whose first 256 bytes now take the part's row scales in planar order (sLc
        // of the 32 tokens, then sRc); lane l reads token l's pair
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        const float2 sa = reinterpret_cast<const float2*>(sm + OFF_SCR + sc * TILE * 8)[part * PART + lane];
        reinterpret_cast<float*>(stg_p)[lane] = sa.x;
        reinterpret_cast<float*>(stg_p)[PART + lane] = sa.y;
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_SEMPTY]);
        // u = sLc S_L + sRc S_R in token pairs (the scales by broadcast loads: every
        // lane reads the same 16 bytes)
        const float4* sl4 = reinterpret_cast<const float4*>(stg_p);
        const float4* sr4 = reinterpret_cast<const float4*>(stg_p + PART * 4);
        uint64_t u2[PART / 2];
#pragma unroll
        for (int k = 0; k < PART / 4; ++k) {  // tokens 4k .. 4k + 3
          const float4 l4 = sl4[k], r4 = sr4[k];
          const int j = 2 * k;
          u2[j] = fma2(pk2(r4.x, r4.y), pk2(__uint_as_float(rr[2 * j]), __uint_as_float(rr[2 * j + 1])),
                       mul2(pk2(l4.x, l4.y), pk2(__uint_as_float(rl[2 * j]), __uint_as_float(rl[2 * j + 1]))));
          u2[j + 1] = fma2(pk2(r4.z, r4.w), pk2(__uint_as_float(rr[2 * j + 2]), __uint_as_float(rr[2 * j + 3])),
                           mul2(pk2(l4.z, l4.w), pk2(__uint_as_float(rl[2 * j + 2]), __uint_as_float(rl[2 * j + 3]))));
        }
        // tokens without data (a suffix of the part, in a partial tile) get -inf
        if (my_n < PART) {
#pragma unroll
          for (int j = 0; j < PART / 2; ++j) {
            const float2 v = up2(u2[j]);
            u2[j] = pk2(2 * j < my_n ? v.x : -INFINITY, 2 * j + 1 < my_n ? v.y : -INFINITY);
          }
        }
        float umax = -INFINITY;
#pragma unroll
        for (int j = 0; j < PART / 2; ++j) {
          const float2 v = up2(u2[j]);
          umax = max3(umax, v.x, v.y);
        }
        // the part's largest row scale: lane l holds token l of the part
        float smax = lane < my_n ? sa.x : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        // tile maxima (score of this head, and row scale) over the four parts
        xmax[(buf * 4 + part) * HG + hh] = umax;
        if (lane == 0) xsm[(buf * 4 + part) * 4 + q] = smax;
        if (!quarter_sync()) {
          ok = false;
          break;
        }
        const float* xm = xmax + buf * 4 * HG + hh;
        const float umax_t = fmaxf(fmaxf(xm[0], xm[HG]), fmaxf(xm[2 * HG], xm[3 * HG]));
        const float* xs = xsm + buf * 16 + q;
        smax = fmaxf(fmaxf(xs[0], xs[4]), fmaxf(xs[8], xs[12]));
        const float tmax = (c > 0.f) ? c * umax_t : -INFINITY;
        float mn = mu;
        if (tmax > mu + TAU) {
          mn = tmax;
        } else if (tmax < mu - DOWN && tmax >= mhi - DOWN_CAP && tmax > -INFINITY) {
          mn = tmax;  // far below: move down so that this bulk stays inside the e4m3 range
        }
        const float alpha = (mn == mu) ? 1.f : (mu == -INFINITY ? 0.f : ex2_approx(mu - mn));
        mu = mn;
        mhi = fmaxf(mhi, mu);
        const float sref_new = (smax > sref * TAU_S) ? smax : sref;
        const float beta = (sref_new == sref) ? 1.f : (sref > 0.f ? sref / sref_new : 0.f);
        sref = sref_new;
        const float fcol = alpha * beta;
        lsum *= alpha;
        const float wk = sref > 0.f ? P_TOP / sref : 0.f;
        // p = 2^(c u - m) as f16 pairs; a padding head takes c = 1 and m = +inf, so
        // that its weights are 0 (as are those of tokens without data: u = -inf)
        const uint64_t c2 = live ? pk2(c, c) : pk2(1.f, 1.f);
        const float mneg = live ? -fmaxf(mu, -3.0e38f) : -INFINITY;
        const uint64_t m2 = pk2(mneg, mneg);
        uint32_t ph[PART / 2];
        uint64_t ls2 = pk2(0.f, 0.f);  // running sums of the even and the odd tokens
#pragma unroll
        for (int j = 0; j < PART / 2; ++j) {
          const float2 z = up2(fma2(c2, u2[j], m2));
          const float p0 = ex2_approx(z.x), p1 = ex2_approx(z.y);
          ls2 = add2(ls2, pk2(p0, p1));
          const __half2 h2 = __floats2half2_rn(p0, p1);
          ph[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        {
          const float2 ls = up2(ls2);
          lsum += ls.x + ls.y;
        }
        // the part's token weights w_t = sLc_t P_TOP / s_ref (0 without data): lane l
        // takes token l
        const float wt = (lane < my_n) ? sa.x * wk : 0.f;
        // the context CTA must be done with this payload buffer's previous tile
        if (i >= 2 &&
            !mbar_wait_warp(&bars[B_PFREE + pb], ((i >> 1) + 1) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        // the payload goes to the staging chunk (its previous copy was waited for
        // at the top of the tile)
#pragma unroll
        for (int u16 = 0; u16 < 4; ++u16)
          sts128(stg + C_P16 + prow(lane, u16),
                 make_uint4(ph[4 * u16], ph[4 * u16 + 1], ph[4 * u16 + 2], ph[4 * u16 + 3]));
        reinterpret_cast<float*>(stg_p + C_FCOL)[lane] = fcol;
        reinterpret_cast<__half*>(stg_p + C_W)[lane] = __float2half_rn(wt);
        if (lane == 0)
          *reinterpret_cast<uint4*>(stg_p + C_EXTRA) = make_uint4(__float_as_uint(sref), 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          bulk_copy_to_cta(prem + pb * P_STRIDE, stg, (uint32_t)CHUNK, pfull_rem + pb * 8);
          bulk_commit();
        }
        __syncwarp();
      }
      if (!ok) {
        fail();
      } else {
        // denominators over the four parts; the partial's (m, l) per head
        xl[part * HG + hh] = lsum;
        if (quarter_sync()) {
          if (part == 0 && h0 + hh < a.H) {
            const int64_t base = item * HG;
            a.ws_m[base + hh] = mu;
            a.ws_l[base + hh] = (xl[hh] + xl[HG + hh]) + (xl[2 * HG + hh] + xl[3 * HG + hh]);
          }
        } else {
          fail();
        }
      }
      // the copies have left this CTA, and the context CTA's last commits to this
      // CTA's barriers have landed
      if (lane == 0) bulk_wait_all();
      if (ok && warp == W_LANE && lane == 0) {
        const int zero = 0;
        for (int i = (n_tiles > 2 ? n_tiles - 2 : 0); i < n_tiles; ++i)
          (void)mbar_wait(&bars[B_PFREE + (i & 1)], (i >> 1) & 1, &zero, WAIT_NS);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ context CTA
    const uint32_t pbuf = smem_u32(sm + OFF_P);
    const uint32_t vring = smem_u32(sm + OFF_VRING);
    if (warp == W_TMA) {
      // The whole warp walks the loop and waits; one elected lane issues.
      int32_t* pt = reinterpret_cast<int32_t*>(sm + OFF_PT);
      load_page_table(a, b, t0, t_end, pt, lane);
      bool ok = true;
      int nv = 0;  // tiles requested
      for (int i = 0; ok && i < n_tiles; ++i) {
        const TileRows tr = tile_rows(a, b, t0, t_end, i, pt);
        const int vs = i % NVT;
        if (!mbar_wait_warp(&bars[B_VEMPTY + vs], ((i / NVT) & 1) ^ 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        facts[vs] = pack_facts(tr);  // released by the arrive below (every lane, one word)
        mbar_arrive_expect_tx_warp(&bars[B_VT + vs],
                                   4u * ((tr.s0 >= 0 ? 8192u : 0u) + (tr.s1 >= 0 ? 8192u : 0u)));
        for (int m = 0; m < 4; ++m) {
          const uint32_t dst = vring + vs * VTILE + m * KBLK;
          if (tr.s0 >= 0) tma_load_2d_warp(dst, &kmap, 128 * m, (int)tr.s0, &bars[B_VT + vs]);
          if (tr.s1 >= 0) tma_load_2d_warp(dst + 8192, &kmap, 128 * m, (int)tr.s1, &bars[B_VT + vs]);
        }
        ++nv;
      }
      if (!ok) {
        if (lane == 0) fail();
        const int zero = 0;
        for (int i = (nv > NVT ? nv - NVT : 0); i < nv; ++i)
          (void)mbar_wait(&bars[B_VT + i % NVT], (i / NVT) & 1, &zero, WAIT_NS);
      }
      __syncwarp();
    } else if (warp == W_MMA) {
      // The whole warp walks the loop and waits; one elected lane issues.
      const uint32_t idV = idesc_f16(128, 256, false, true);  // A = P'' K-major, B = V MN-major
      const uint64_t pdesc = smem_desc(pbuf, 16, 1024, SW128);
      const uint64_t vdesc = smem_desc(vring, KBLK, 1024, SW128);
      bool ok = true;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int pb = i & 1, vs = i % NVT;
        for (int half = 0; half < 2; ++half) {
          // operand, V rows and this O half ready (the lane workers' barrier)
          if (!mbar_wait_warp(&bars[B_RS + half], i & 1, abort_flag, WAIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = pdesc + (uint64_t)((pb * P_STRIDE) >> 4);
          const uint64_t bd = vdesc + (uint64_t)((vs * VTILE + half * 2 * KBLK) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: 32 tokens of the hi / lo atom (32 bytes in); B: 32 token rows of V (4 KB in)
            mma_f8_warp(tmem + half * 256, ad + 2 * kk, bd + 256 * kk, idV, (i > 0 || kk > 0) ? 1u : 0u);
            mma_f8_warp(tmem + half * 256, ad + (KBLK >> 4) + 2 * kk, bd + 256 * kk, idV, 1u);
          }
          mma_commit_warp(&bars[B_ODONE + half]);
        }
        if (!ok) break;
        mma_commit_warp(&bars[B_VEMPTY + vs]);
        mma_commit_mc_warp(&bars[B_PFREE + pb], (uint16_t)0x3);
      }
      if (!ok && lane == 0) fail();
      const int zero = 0;
      mma_commit_warp(&bars[B_DRAIN]);
      (void)mbar_wait(&bars[B_DRAIN], 0, &zero, WAIT_NS);
      __syncwarp();
    } else {
      // ---------------------------------------------------------- operand, V rows,
      // O rescale and epilogue
      const int q = warp & 3;
      const int part = (warp - W_LANE) >> 2;   // part of the tile / 64 columns of an O half
      const int hh = q * 32 + lane;
      const int chunk = part * 4 + q;          // the payload chunk of these heads and tokens
      const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
      bool ok = true;
      float sref_fin = 0.f;
      int cvt_phase = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int pb = i & 1, vs = i % NVT;
        if (!mbar_wait_warp(&bars[B_PFULL + pb], (i >> 1) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        // this thread's row of the payload (p for 32 tokens of head hh), the head's
        // rescale factor and the part's token weights (as f16 pairs)
        const uint32_t cb = pbuf + pb * P_STRIDE + chunk * CHUNK;
        const uint8_t* cp = sm + OFF_P + pb * P_STRIDE + chunk * CHUNK;
        uint4 pv[4];
#pragma unroll
        for (int u16 = 0; u16 < 4; ++u16) pv[u16] = lds128(cb + C_P16 + prow(lane, u16));
        const float f = reinterpret_cast<const float*>(cp + C_FCOL)[lane];
        if (i == n_tiles - 1) sref_fin = reinterpret_cast<const float*>(cp + C_EXTRA)[0];
        uint32_t wh[PART / 2];
#pragma unroll
        for (int k = 0; k < PART / 8; ++k) {
          const uint4 w8 = lds128(cb + C_W + 16 * k);  // f16 weights of tokens 8k .. 8k + 7
          wh[4 * k] = w8.x;
          wh[4 * k + 1] = w8.y;
          wh[4 * k + 2] = w8.z;
          wh[4 * k + 3] = w8.w;
        }
        const bool any = __any_sync(0xffffffffu, f != 1.f) && i > 0;
        // every warp has read this payload: its buffer may now take the operand
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_CVT]);
        if (!mbar_wait_warp(&bars[B_CVT], (cvt_phase++) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        // the buffer's next payload (tile i + 2) may only be expected once this one
        // has been read; its bytes come after the context MMAs of tile i
        if (warp == W_LANE && lane == 0 && i + 2 < n_tiles)
          mbar_arrive_expect_tx(&bars[B_PFULL + pb], (uint32_t)P_BYTES);
        // P''[h][t] = p w_t in f16, as two e4m3 terms, into the hi and lo atoms
        // (K-major, 128-byte swizzle) of the same buffer
        const uint32_t opnd = pbuf + pb * P_STRIDE;
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // 16 tokens per 16-byte unit
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = 16 * j + 4 * k;  // tokens t .. t + 3: two f16 pairs of p and of w
            const uint4 src = pv[t / 8];
            const uint32_t p01 = (t % 8 == 0) ? src.x : src.z, p23 = (t % 8 == 0) ? src.y : src.w;
            const __half2 x01 = __hmul2(*reinterpret_cast<const __half2*>(&p01),
                                        *reinterpret_cast<const __half2*>(&wh[t / 2]));
            const __half2 x23 = __hmul2(*reinterpret_cast<const __half2*>(&p23),
                                        *reinterpret_cast<const __half2*>(&wh[t / 2 + 1]));
            uint16_t h01, l01, h23, l23;
            split_h2(x01, h01, l01);
            split_h2(x23, h23, l23);
            hw[k] = (uint32_t)h01 | ((uint32_t)h23 << 16);
            lw[k] = (uint32_t)l01 | ((uint32_t)l23 << 16);
          }
          const uint32_t off = sw128(hh, part * 2 + j);
          sts128(opnd + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
          sts128(opnd + KBLK + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
        }
        // V tile: rows without data (past the item, or a page that is absent or
        // unmapped) are zeroed so that their zero weights meet no NaN; warp w takes
        // rows r = w (mod 16), a lane one 16-byte unit of one d-block
        if (!mbar_wait_warp(&bars[B_VT + vs], (i / NVT) & 1, abort_flag, WAIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t vf = facts[vs];
        if (vf != FULL_TILE) {
          const uint32_t vb = vring + vs * VTILE;
          for (int r = warp - W_LANE; r < TILE; r += N_LANE_WARPS)
            if (!row_has(vf, r))
              sts128(vb + (lane >> 3) * KBLK + r * 128 + (lane & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
        // Each O half: the previous tile's MMAs on it are done (waited for on every
        // tile, rescale or not: the operand-ready barrier of this half then runs at
        // most one phase ahead of the MMA thread that waits on it), then the rows of
        // heads whose factor moved are rescaled, then the half is released.
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          if (i > 0 &&
              !mbar_wait_warp(&bars[B_ODONE + half], (i - 1) & 1, abort_flag, WAIT_NS)) {
            ok = false;
            break;
          }
          if (any) {
            tc_fence_after();
            __syncwarp();
            const uint32_t col = tmem + lane_addr + half * 256 + part * 64;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 16) {
              uint32_t r[16];
              tmem_ld16(col + c0, r);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * f);
              tmem_st16(col + c0, r);
            }
            __syncwarp();
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_RS + half]);
        }
        if (!ok) break;
      }
      if (ok) {
        ok = mbar_wait_warp(&bars[B_ODONE], (n_tiles - 1) & 1, abort_flag, WAIT_NS) &&
             mbar_wait_warp(&bars[B_ODONE + 1], (n_tiles - 1) & 1, abort_flag, WAIT_NS);
      }
      if (ok) {
        // epilogue: the partial's unnormalised o = acc * s_ref / P_TOP.  A thread's
        // TMEM lane is one head: it puts its head's 64 columns of an O half in a
        // shared-memory row (the payload buffers and V ring, free now; rows 272
        // bytes apart, so a quarter warp's 16-byte stores fall on distinct banks) and
        // sends the row to the workspace with one 256-byte bulk copy.
        tc_fence_after();
        __syncwarp();
        const float oscale = sref_fin * (1.0f / P_TOP);
        const uint32_t stage = smem_u32(sm + OFF_P) + (uint32_t)(warp - W_LANE) * (32 * O_ROW);
        const bool real = h0 + q * 32 + lane < a.H;
        float* dst = a.ws_o + (item * HG + q * 32 + lane) * DL;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          const int cbase = half * 256 + part * 64;
          if (half > 0) {
            bulk_wait_read_all();  // this lane's row of the first half has been read
            __syncwarp();
          }
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_addr + cbase + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              sts128(stage + lane * O_ROW + (c0 + k) * 4,
                     make_uint4(__float_as_uint(__uint_as_float(r[k]) * oscale),
                                __float_as_uint(__uint_as_float(r[k + 1]) * oscale),
                                __float_as_uint(__uint_as_float(r[k + 2]) * oscale),
                                __float_as_uint(__uint_as_float(r[k + 3]) * oscale)));
          }
          fence_proxy_async_smem();
          if (real) {
            bulk_store_s2g(dst + cbase, stage + lane * O_ROW, 64 * 4);
            bulk_commit();
          }
        }
        bulk_wait_all();  // the rows have landed before the CTA leaves
      } else {
        fail();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while its partner may still write to it
  tc_fence_after();
  if (warp == W_MMA) tmem_dealloc(tmem, 512);
}

// The queries in the score operand's form, one warp per (sequence, head): a
// power-of-two scale 2^e puts max|q| over the 576 channels in [128, 256), each
// scaled value becomes two e4m3 terms, hi = e4m3(x) and lo = e4m3(x - hi), and
// c_h = sm_scale * log2(e) / 2^e undoes the scale in the softmax.  Bytes of a head:
// Lc hi (channel order), Lc lo, Rc hi, Rc lo.
__global__ void __launch_bounds__(256) prep_query_kernel(const DecodeArgs a) {
  grid_dependents_launch();  // the decode kernel's set-up may overlap this launch
  const int64_t head = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // b * H + h
  if (head >= (int64_t)a.B * a.H) return;
  const int lane = threadIdx.x & 31;
  const float4* ql = reinterpret_cast<const float4*>(a.q_lat + head * DL);
  const float4* qr = reinterpret_cast<const float4*>(a.q_rope + head * DR);
  float4 x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = __ldg(ql + 32 * k + lane);  // channels 4 (32 k + lane) + 0..3
  const float4 y = lane < 16 ? __ldg(qr + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  float amax = fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w)));
#pragma unroll
  for (int k = 0; k < 4; ++k)
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int e = 0;
  if (amax > 0.f && isfinite(amax)) {
    int ex;
    frexpf(amax, &ex);
    e = min(max(8 - ex, -120), 120);
  }
  const float sc = ldexpf(1.0f, e);
  uint32_t* dst = reinterpret_cast<uint32_t*>(a.q8 + head * Q8_BYTES);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float v[4] = {x[k].x * sc, x[k].y * sc, x[k].z * sc, x[k].w * sc};
    uint32_t hi, lo;
    split4(v, hi, lo);
    dst[32 * k + lane] = hi;
    dst[DL / 4 + 32 * k + lane] = lo;
  }
  if (lane < 16) {
    const float v[4] = {y.x * sc, y.y * sc, y.z * sc, y.w * sc};
    uint32_t hi, lo;
    split4(v, hi, lo);
    dst[2 * DL / 4 + lane] = hi;
    dst[2 * DL / 4 + DR / 4 + lane] = lo;
  }
  if (lane == 0) a.cq[head] = a.sm_scale * LOG2E / sc;
}

}  // namespace

cudaError_t launch_prep_query(const DecodeArgs& a, cudaStream_t s) {
  if (a.q8 == nullptr || a.cq == nullptr) return cudaErrorInvalidValue;  // no room planned for them
  const int64_t heads = (int64_t)a.B * a.H;
  if (heads > 0) prep_query_kernel<<<(unsigned)((heads + 7) / 8), 256, 0, s>>>(a);
  return cudaGetLastError();
}

// Pairs that can be resident at once (clusters of two on this device).
cudaError_t pair_capacity(int* pairs) {
  static std::atomic<int> memo[MAX_DEVICES];
  return per_device(memo, [](int* v) {
    cudaError_t r = cudaFuncSetAttribute(decode_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (r != cudaSuccess) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NUM_SMS, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    int n = 0;
    r = cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel, &cfg);
    if (r != cudaSuccess) return r;
    if (n < 1) return cudaErrorLaunchOutOfResources;  // no pair fits: say so, never plan for one
    *v = n > NUM_SMS / 2 ? NUM_SMS / 2 : n;
    return cudaSuccess;
  }, pairs);
}

cudaError_t launch_decode_pair(const DecodeArgs& a, cudaStream_t s) {
  if (a.plan.hg != HG) return cudaErrorNotSupported;
  int pairs = 0;
  cudaError_t e = pair_capacity(&pairs);
  if (e != cudaSuccess) return e;
  // the items are cut for the pairs this device holds at once (never more than
  // the plan's bound, so the workspace the plan sized still holds every item)
  DecodeArgs d = a;
  if (pairs < d.plan.target) d.plan.target = pairs;
  CUtensorMap kmap, smap;
  e = make_cache_map(d, &kmap);
  if (e != cudaSuccess) return e;
  e = make_scale_map(d, &smap);
  if (e != cudaSuccess) return e;
  e = launch_prep_query(d, s);
  if (e != cudaSuccess) return e;
  return launch_after_prep(decode_pair_kernel, 2 * d.plan.max_items, NTHREADS, SMEM, s, d, kmap, smap);
}

}  // namespace kv8
