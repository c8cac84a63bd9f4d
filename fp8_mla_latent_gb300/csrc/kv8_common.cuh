// kv8_common.cuh -- small device helpers shared by the kernels of libfp8mla.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kv8_internal.h"

namespace kv8 {

// Two e4m3 bytes (low byte = element 0) -> two fp16 values, exactly (every
// e4m3 value, subnormals included, is an fp16 value).  Hardware cvt on sm_89+.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("{ cvt.rn.f16x2.e4m3x2 %0, %1; }" : "=r"(r) : "h"(v));
  return r;
}

// Four e4m3 bytes -> four floats (exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  const uint32_t lo = e4m3x2_to_f16x2((uint16_t)(w & 0xFFFFu));
  const uint32_t hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// Two floats -> two e4m3 bytes (element 0 in the low byte), round to nearest
// even, finite results saturate at +-448.  Callers remove NaN first.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float e0, float e1) {
  uint16_t r;
  // the first source operand lands in the upper byte
  asm("{ cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2; }" : "=h"(r) : "f"(e1), "f"(e0));
  return r;
}

// f16x2 -> two e4m3 bytes (the low half lands in the low byte), round to
// nearest even, finite results saturate at +-448.
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(__half2 v) {
  uint16_t r;
  asm("{ cvt.rn.satfinite.e4m3x2.f16x2 %0, %1; }" : "=h"(r) : "r"(*reinterpret_cast<const uint32_t*>(&v)));
  return r;
}

// Length of sequence b, clamped to what its block table can address.
__device__ __forceinline__ int64_t seq_len_of(const DecodeArgs& a, int b) {
  if (a.seq_lens == nullptr) return a.T_contig;
  int64_t T = __ldg(&a.seq_lens[b]);
  const int64_t cap = (int64_t)a.max_blocks * PAGE;
  if (T < 0 || T > cap) {
    atomicOr(a.err, ERR_SEQ_LEN);
    T = T < 0 ? 0 : cap;
  }
  return T;
}

// ---------------------------------------------------------------------------
// Work items of a decode call.  The tokens of every (sequence, head group) are
// cut into items of `st` tiles: st is the smallest item length whose items all
// fit in one wave of `target` CTAs (so no CTA waits for a second wave behind a
// long item), and never below ceil(total tiles x head groups / target).  When
// there are more (sequence, head group) pairs than one wave holds, the items are
// ceil(total / target) tiles long and spread over several waves.  Items are
// numbered by sequence, then head group, then position; every kernel of a call
// derives the same numbering from the sequence lengths, on the device.  The
// tensor-core kernels count in 128-token tiles; the CUDA-core kernel in 32-token
// units, so that a short cache spreads over more SMs.

struct WorkItem {
  int b, g;        // sequence, head group
  int64_t t0, t1;  // tokens [t0, t1) of sequence b
  int64_t first, count;  // items of (b, g): [first, first + count)
};

// The CTA of the first item of (b, g) records that segment for the merge.
__device__ __forceinline__ void record_segment(const DecodeArgs& a, int64_t k, const WorkItem& it) {
  if (k == it.first) {
    int64_t* e = a.seg + ((int64_t)it.b * a.plan.n_hg + it.g) * 2;
    e[0] = it.first;
    e[1] = it.count;
  }
}

__device__ __forceinline__ uint32_t tiles_of(const DecodeArgs& a, int b, int lg = LOG2_TILE) {
  // a length is at most max_blocks * PAGE (or the contiguous cache's rows, below
  // 2^31), so the count of 128-token tiles fits 32 bits
  return (uint32_t)((seq_len_of(a, b) + (int64_t(1) << lg) - 1) >> lg);
}

// Tile counts of the sequences, held in registers: lane l keeps sequences l,
// l + 32, ... (SEQ_CACHE of them).  With more than 32 * SEQ_CACHE sequences
// nothing is kept and the counts are read again from seq_lens at every use.
// (The item plan is found by a search that counts items for several lengths:
// from registers, in 32-bit arithmetic, that costs each CTA about a microsecond
// at the start of a call instead of several.)
constexpr int SEQ_CACHE = 4;
struct SeqTiles {
  uint32_t t[SEQ_CACHE];  // units of 2^lg tokens (tiles, unless a kernel cuts finer)
  uint32_t n[SEQ_CACHE];  // tokens (clamped lengths, below 2^31)
  int lg;
  bool cached;
};

// Warp-wide (all 32 lanes).
__device__ __forceinline__ void load_tiles(const DecodeArgs& a, SeqTiles& c, int lg = LOG2_TILE) {
  const int lane = threadIdx.x & 31;
  c.lg = lg;
  c.cached = a.B <= 32 * SEQ_CACHE;
#pragma unroll
  for (int k = 0; k < SEQ_CACHE; ++k) {
    const int b = lane + 32 * k;
    const uint32_t n = (c.cached && b < a.B) ? (uint32_t)seq_len_of(a, b) : 0u;
    c.n[k] = n;
    c.t[k] = (n + ((1u << lg) - 1u)) >> lg;
  }
}

// Length of sequence 32 k + lane (0 past the last sequence).
__device__ __forceinline__ uint32_t len_at(const DecodeArgs& a, const SeqTiles& c, int k) {
  if (c.cached) {
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < SEQ_CACHE; ++j) v = (j == k) ? c.n[j] : v;
    return v;
  }
  const int b = 32 * k + (int)(threadIdx.x & 31);
  return b < a.B ? (uint32_t)seq_len_of(a, b) : 0u;
}

// Tiles of sequence 32 k + lane (0 past the last sequence).
__device__ __forceinline__ uint32_t tiles_at(const DecodeArgs& a, const SeqTiles& c, int k) {
  if (c.cached) {
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < SEQ_CACHE; ++j) v = (j == k) ? c.t[j] : v;
    return v;
  }
  const int b = 32 * k + (int)(threadIdx.x & 31);
  return b < a.B ? tiles_of(a, b, c.lg) : 0u;
}

__device__ __forceinline__ uint64_t warp_sum64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Warp-wide: number of items if every sequence is cut into pieces of st tiles
// (1 <= st < 2^31), times the head groups.
__device__ __forceinline__ int64_t count_items(const DecodeArgs& a, const SeqTiles& c, uint32_t st) {
  uint64_t n = 0;
  if (c.cached) {
#pragma unroll
    for (int k = 0; k < SEQ_CACHE; ++k) {
      if (32 * k >= a.B) break;
      n += (c.t[k] + (st - 1u)) / st;
    }
  } else {
    for (int k = 0; 32 * k < a.B; ++k) {
      const uint32_t t = tiles_at(a, c, k);
      n += (t + (st - 1u)) / st;
    }
  }
  return (int64_t)warp_sum64(n) * a.plan.n_hg;
}

// Warp-wide: tiles per item for this call.  The search evaluates the item count
// at one probe per pass (lo, then the longest sequence, then bisection), so the
// count is inlined once: this runs once per CTA, and its code size, not its
// arithmetic, is what it costs.
__device__ __forceinline__ int64_t item_tiles(const DecodeArgs& a, const SeqTiles& c) {
  uint64_t total = 0;
  uint32_t tmax = 0;
  for (int k = 0; 32 * k < a.B; ++k) {
    const uint32_t t = tiles_at(a, c, k);
    total += t;
    tmax = t > tmax ? t : tmax;
  }
  total = warp_sum64(total);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t m = __shfl_xor_sync(0xffffffffu, tmax, o);
    tmax = m > tmax ? m : tmax;
  }
  const int64_t jobs = (int64_t)total * a.plan.n_hg;
  int64_t lo = (jobs + a.plan.target - 1) / a.plan.target;
  if (lo < 1) lo = 1;
  if ((int64_t)tmax <= lo) return lo;
  // lo < tmax < 2^31 from here.  Invariant once bisecting: count(l) > target >=
  // count(h); the count falls as the item length grows.
  uint32_t l = (uint32_t)lo, h = tmax, probe = l;
  int pass = 0;
#pragma unroll 1
  for (;;) {
    const bool fits = count_items(a, c, probe) <= a.plan.target;
    if (pass == 0) {
      if (fits) return lo;
      pass = 1;
      probe = h;
      continue;
    }
    if (pass == 1) {
      if (!fits) return lo;  // more pairs than one wave holds
      pass = 2;
    } else if (fits) {
      h = probe;
    } else {
      l = probe;
    }
    if (l + 1 >= h) return h;
    probe = l + (h - l) / 2;
  }
}

// Warp-wide: the work item with index k; false if k is past the last item.  Items
// are whole units of 2^lg tokens (tiles, unless a kernel asks for finer cuts).  The
// sequences are walked 32 at a time with the inclusive scan of their item counts.
// Item counts and indices fit 32 bits (the grid holds every item), and so does a
// sequence's tile count; only token offsets need 64 bits.
__device__ __forceinline__ bool find_item(const DecodeArgs& a, int64_t k, WorkItem& it,
                                          int lg = LOG2_TILE) {
  const int lane = threadIdx.x & 31;
  SeqTiles c;
  load_tiles(a, c, lg);
  const int64_t st = item_tiles(a, c);
  // st >= 2^31 only when every sequence is one item: ceil(tiles / st) is then 0 or 1
  const uint32_t st32 = st < (int64_t(1) << 31) ? (uint32_t)st : 0x80000000u;
  const uint32_t k32 = (uint32_t)k, n_hg = (uint32_t)a.plan.n_hg;
  uint32_t base = 0;
  for (int kk = 0; 32 * kk < a.B; ++kk) {
    const int b = 32 * kk + lane;
    const uint32_t tiles = tiles_at(a, c, kk);
    const uint32_t ns = tiles / st32 + (tiles % st32 != 0u ? 1u : 0u);
    const uint32_t cnt = ns * n_hg;
    uint32_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const uint32_t first = base + inc - cnt;
    const bool mine = (b < a.B) && k32 >= first && k32 < first + cnt;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (m) {
      const int src = __ffs(m) - 1;
      const int bb = __shfl_sync(0xffffffffu, b, src);
      const uint32_t fb = __shfl_sync(0xffffffffu, first, src);
      const uint32_t nsb = __shfl_sync(0xffffffffu, ns, src);
      const uint32_t r = k32 - fb;
      const uint32_t s = r % nsb;
      it.b = bb;
      it.g = (int)(r / nsb);
      it.t0 = ((int64_t)s * st) << lg;
      const int64_t T = __shfl_sync(0xffffffffu, len_at(a, c, kk), src);
      const int64_t e = ((int64_t)(s + 1) * st) << lg;
      it.t1 = e < T ? e : T;
      it.first = (int64_t)fb + (int64_t)it.g * nsb;
      it.count = nsb;
      return true;
    }
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  return false;
}

// ---------------------------------------------------------------------------
// Ranges for the one-CTA tensor-core kernel.  The tiles of all (sequence, head
// group) pairs, pair after pair, are cut into NC = min(target, total) ranges of
// equal length (to one tile), one per CTA; a range may run from the end of one
// pair's tiles into the start of the next.  This is used when every nonempty
// pair has at least a range's worth of tiles (a range then holds at most two
// segments) and when the per-sequence items would be longer than a range (64
// sequences of 64 tiles on 152 SMs: items of 32 tiles against ranges of 27).
// Segments are numbered in order, so the segments of a pair are consecutive and
// the merge reads them as it reads items.

struct Segment {
  int b, g;
  int64_t t0, t1;        // tokens [t0, t1) of sequence b
  int64_t sid;           // partial index
  int64_t first, count;  // the pair's segments (meaningful where starts)
  bool starts;           // the pair's first segment
};
struct Range {
  int n;                 // segments: 0 (no work), 1 or 2
  Segment s[2];
};

// First tile of range k of NC over `total` tiles, and the range holding tile x
// (s32: total * NC < 2^32, so every product and quotient fits 32 bits).
__device__ __forceinline__ int64_t range_start(int64_t k, int64_t NC, int64_t total, bool s32) {
  return s32 ? (int64_t)((uint32_t)(k * total) / (uint32_t)NC) : k * total / NC;
}
__device__ __forceinline__ int64_t range_of(int64_t x, int64_t NC, int64_t total, bool s32) {
  return s32 ? (int64_t)((uint32_t)((x + 1) * NC - 1) / (uint32_t)total) : ((x + 1) * NC - 1) / total;
}

// Warp-wide: whether this call runs on ranges, and if so CTA k's range.  Returns
// false when the per-sequence items (find_item) apply instead.
__device__ __forceinline__ bool find_range(const DecodeArgs& a, int64_t k, Range& r) {
  const int lane = threadIdx.x & 31;
  SeqTiles c;
  load_tiles(a, c);
  const int n_hg = a.plan.n_hg;
  uint64_t total = 0;
  uint32_t tmin = 0xFFFFFFFFu;
  for (int kk = 0; 32 * kk < a.B; ++kk) {
    const uint32_t t = tiles_at(a, c, kk);
    total += t;
    if (t > 0u && t < tmin) tmin = t;
  }
  total = warp_sum64(total) * (uint64_t)n_hg;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t m = __shfl_xor_sync(0xffffffffu, tmin, o);
    tmin = m < tmin ? m : tmin;
  }
  if (total == 0) return false;
  const int64_t NC = (int64_t)total < a.plan.target ? (int64_t)total : a.plan.target;
  const int64_t L = ((int64_t)total + NC - 1) / NC;
  // the per-sequence items' length exceeds L exactly when items of L tiles do not
  // fit in one wave (the count falls as the length grows, and L >= the lower
  // bound of that search)
  if ((int64_t)tmin < L || count_items(a, c, (uint32_t)L) <= a.plan.target) return false;
  r.n = 0;
  if (k >= NC) return true;  // no range for this CTA
  const bool s32 = total * (uint64_t)NC < (uint64_t(1) << 32);
  const int64_t T0 = range_start(k, NC, total, s32), T1 = range_start(k + 1, NC, total, s32);
  // Walk the pairs in order: the pair holding T0 (segment 0), the next one if
  // the range reaches it (segment 1), and the pair starts before T0 that do not
  // fall on a range start (each adds a segment to the numbering).
  int64_t base = 0, extra = 0;
  int found = 0;
  for (int kk = 0; 32 * kk < a.B; ++kk) {
    const int b = 32 * kk + lane;
    const int64_t tl = tiles_at(a, c, kk);
    const int64_t len = tl * n_hg;
    int64_t inc = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const int64_t sb = base + inc - len;  // first tile of sequence b's pairs
    int cnt = 0;
    for (int g = 0; g < n_hg && tl > 0; ++g) {
      const int64_t st = sb + g * tl;
      if (st > 0 && st < T0 && range_start(range_of(st, NC, total, s32), NC, total, s32) != st) ++cnt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    extra += cnt;
    // the sequences holding T0 and T1 - 1
    for (int want = found; want < 2; ++want) {
      const int64_t x = want == 0 ? T0 : T1 - 1;
      const bool mine = (b < a.B) && tl > 0 && x >= sb && x < sb + len;
      const unsigned m = __ballot_sync(0xffffffffu, mine);
      if (!m) break;
      const int src = __ffs(m) - 1;
      const int bb = __shfl_sync(0xffffffffu, b, src);
      const int64_t sbb = __shfl_sync(0xffffffffu, sb, src), tlb = __shfl_sync(0xffffffffu, tl, src);
      const int g = s32 ? (int)((uint32_t)(x - sbb) / (uint32_t)tlb) : (int)((x - sbb) / tlb);
      const int64_t ps = sbb + g * tlb, pe = ps + tlb;  // the pair's tiles [ps, pe)
      Segment& sg = r.s[want];
      sg.b = bb;
      sg.g = g;
      const int64_t lo = (want == 0 ? T0 : ps) - ps;
      const int64_t hi = (T1 < pe ? T1 : pe) - ps;
      const int64_t T = __shfl_sync(0xffffffffu, len_at(a, c, kk), src);
      sg.t0 = lo * TILE;
      sg.t1 = hi * TILE < T ? hi * TILE : T;
      sg.starts = (lo == 0);
      sg.first = 0;  // set below, with the numbering
      sg.count = range_of(pe - 1, NC, total, s32) - range_of(ps, NC, total, s32) + 1;
      found = want + 1;
    }
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  // segment 1 exists when the range ends in another pair than it starts in
  r.n = (found == 2 && (r.s[1].b != r.s[0].b || r.s[1].g != r.s[0].g)) ? 2 : 1;
  r.s[0].sid = k + extra;
  r.s[1].sid = k + extra + 1;
  r.s[0].first = r.s[0].sid;
  r.s[1].first = r.s[1].sid;
  return true;
}

// The CTA holding a pair's first segment records the pair's segments for the merge.
__device__ __forceinline__ void record_range_segment(const DecodeArgs& a, const Segment& s) {
  if (s.starts) {
    int64_t* e = a.seg + ((int64_t)s.b * a.plan.n_hg + s.g) * 2;
    e[0] = s.first;
    e[1] = s.count;
  }
}

// ---------------------------------------------------------------------------
// Pages of a work item, for the tensor-core kernels: the item's block-table
// entries are read once into shared memory, and every tile's two pages become
// cache slots (or -1) from there.

constexpr int PT_PAGES = 256;  // block-table entries of an item kept in shared memory

// Per-tile page facts.
struct TileRows {
  int64_t s0, s1;  // cache slot of the tile's first / second page, or -1 (absent or unmapped)
  int nv;          // tokens of the tile inside the item
};
// Cache slot of token t of the item starting at token t0: its block-table entry
// from the item's copy in shared memory (the first PT_PAGES pages), else from global
// memory; -1 (and the error bit) for an entry out of range.
__device__ __forceinline__ int64_t item_slot(const DecodeArgs& a, int b, int64_t t, int64_t t0,
                                             const int32_t* pt) {
  if (a.block_table == nullptr) return t;
  const int64_t k = (t >> 6) - (t0 >> 6);
  const int32_t blk = k < PT_PAGES ? pt[k] : __ldg(&a.block_table[(int64_t)b * a.max_blocks + (t >> 6)]);
  if (blk < 0 || (int64_t)blk >= a.n_blocks) {
    atomicOr(a.err, ERR_BLOCK_TABLE);
    return -1;
  }
  return (int64_t)blk * PAGE + (t & (PAGE - 1));
}
// The item's first PT_PAGES block-table entries into shared memory, by all lanes of
// the calling warp (one round trip instead of a dependent lookup per page).
__device__ __forceinline__ void load_page_table(const DecodeArgs& a, int b, int64_t t0,
                                                int64_t t_end, int32_t* pt, int lane) {
  if (a.block_table != nullptr) {
    const int64_t p0 = t0 >> 6, np = ((t_end + PAGE - 1) >> 6) - p0;
    for (int k = lane; k < PT_PAGES && k < np; k += 32)
      pt[k] = __ldg(&a.block_table[(int64_t)b * a.max_blocks + p0 + k]);
  }
  __syncwarp();
}
__device__ __forceinline__ TileRows tile_rows(const DecodeArgs& a, int b, int64_t t0, int64_t t_end,
                                              int i, const int32_t* pt) {
  TileRows r;
  const int64_t tb = t0 + (int64_t)i * TILE;
  const int64_t n = t_end - tb;
  r.nv = n < TILE ? (int)n : TILE;
  r.s0 = item_slot(a, b, tb, t0, pt);
  r.s1 = r.nv > PAGE ? item_slot(a, b, tb + PAGE, t0, pt) : -1;
  return r;
}
// The facts packed in a word the loading thread leaves in shared memory for the
// warps that read the tile: tokens inside the item (0..128) in bits 0..7, first /
// second page present in bits 8 / 9.
constexpr uint32_t FULL_TILE = TILE | 0x300u;
__device__ __forceinline__ uint32_t pack_facts(const TileRows& r) {
  return (uint32_t)r.nv | (r.s0 >= 0 ? 0x100u : 0u) | (r.s1 >= 0 ? 0x200u : 0u);
}
// row r of the tile holds data
__device__ __forceinline__ bool row_has(uint32_t f, int r) {
  return r < (int)(f & 0xFFu) && ((f >> (8 + r / PAGE)) & 1u) != 0u;
}

// 16-byte shared-memory stores and loads.
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Byte offset of 16-byte unit u of row r in a 128-byte-swizzled K-major atom.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

}  // namespace kv8
