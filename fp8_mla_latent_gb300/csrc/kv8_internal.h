// kv8_internal.h -- launch interface shared by the C-ABI shim and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace kv8 {

constexpr int DL = 512;    // kv_lora latent width
constexpr int DR = 64;     // qk_rope width
constexpr int D = 576;     // bytes per cached row
constexpr int PAGE = 64;   // tokens per page in the paged layout
constexpr int TILE = 128;  // tokens per decode tile (the M of the score MMA)
constexpr int LOG2_TILE = 7;
static_assert((1 << LOG2_TILE) == TILE, "tile size");
constexpr int NUM_SMS = 152;  // GB300: 2 dies x 76 SMs

// Device-side error bits written into the workspace header.
constexpr unsigned ERR_BLOCK_TABLE = 1u;
constexpr unsigned ERR_SEQ_LEN = 2u;
constexpr unsigned ERR_TIMEOUT = 4u;  // a bounded wait in a kernel gave up

// Decode variants (the public kv8_decode_variant values): kTc resolves to the
// SM-pair kernel for H > 64 and to the one-CTA kernel otherwise.
enum Variant { kAuto = 0, kSimt = 1, kTc = 2, kTcCta = 3, kTcPair = 4 };

struct SplitPlan {
  int variant;      // resolved: kSimt, kTcCta or kTcPair
  int hg;           // heads per CTA (head group)
  int n_hg;         // head groups
  int target;       // CTAs the work is spread over (one wave of the split kernel)
  int max_items;    // upper bound on work items: the split kernel's grid size
  int64_t ws_bytes; // workspace bytes needed
  // byte offsets inside the workspace; the header (error word, then the item
  // table) is cleared by every split launch
  int64_t hdr_bytes, off_seg, off_m, off_l, off_o;
  // tensor-core kernels only (0 otherwise): the queries in the score operand's
  // form, written by the query-prep launch: [B][H][Q8_BYTES] e4m3 terms, [B][H] f32 c_h
  int64_t off_q8, off_cq;
};

// Bytes per (sequence, head) of the prepared query: the Lc channels' hi term (512),
// their lo term (512), then the Rc channels' hi (64) and lo (64) terms.
constexpr int Q8_BYTES = 2 * DL + 2 * DR;

// Deterministic in its arguments (no device query), so the workspace-size call
// and the decode call always agree.
SplitPlan plan_decode(int B, int H, int64_t max_len, int variant);

struct DecodeArgs {
  const float* q_lat;          // [B][H][512]
  const float* q_rope;         // [B][H][64]
  const uint8_t* codes;        // [slots][576]
  const float* scales;         // [slots][2]
  const int32_t* block_table;  // [B][max_blocks] or nullptr (contiguous, B == 1)
  const int32_t* seq_lens;     // [B] or nullptr (then T_contig)
  int64_t T_contig;
  int B, H, max_blocks;
  int64_t n_blocks;
  float sm_scale;
  float* out;                  // [B][H][512]
  float* lse;                  // [B][H] or nullptr
  unsigned* err;               // workspace header word
  int64_t* seg;                // [B][n_hg][2]: first work item and item count (0 if none)
  float* ws_m;                 // [max_items][hg]   running max, log2 units
  float* ws_l;                 // [max_items][hg]   sum of exp2(z - m)
  float* ws_o;                 // [max_items][hg][512] unnormalised context
  uint8_t* q8;                 // [B][H][Q8_BYTES] prepared queries (tensor-core kernels), or nullptr
  float* cq;                   // [B][H] their scale factors c_h (tensor-core kernels), or nullptr
  SplitPlan plan;
};

// A launch setting that belongs to the current device (a kernel's shared-memory
// opt-in, an occupancy figure): `make(&v)` computes it (v > 0) the first time a
// device asks; later calls on that device return the stored value.  Settings are
// per device (cudaFuncSetAttribute applies to the current device only), and
// concurrent first calls just compute the same value twice.
constexpr int MAX_DEVICES = 64;
template <typename F>
inline cudaError_t per_device(std::atomic<int> (&memo)[MAX_DEVICES], F&& make, int* value) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return make(value);
  int v = memo[dev].load(std::memory_order_acquire);
  if (v <= 0) {
    e = make(&v);
    if (e != cudaSuccess) return e;
    memo[dev].store(v, std::memory_order_release);
  }
  *value = v;
  return cudaSuccess;
}

// Tensor maps for TMA loads (decode_tc.cu): a tiled map of `rank` dimensions
// (row strides in bytes, rows past the extent read as zeros), the e4m3 cache's
// map (boxes of one 64-row page x 128 bytes, 128-byte swizzle) and the row
// scales' map (1-D, boxes of one page's 128 floats).
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, unsigned rank, void* base,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                         CUtensorMapSwizzle swizzle);
cudaError_t make_cache_map(const DecodeArgs& a, CUtensorMap* map);
cudaError_t make_scale_map(const DecodeArgs& a, CUtensorMap* map);
cudaError_t make_rc_map(const DecodeArgs& a, CUtensorMap* map);

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_pair(const DecodeArgs& a, cudaStream_t s);
// The queries of both tensor-core kernels in their score operand's form (a.q8, a.cq).
cudaError_t launch_prep_query(const DecodeArgs& a, cudaStream_t s);

// Launch of a decode kernel right after the query-prep launch on the same stream,
// as its programmatic dependent: the kernel's set-up overlaps the prep launch, and
// its threads wait (griddepcontrol.wait) before they read the prepared queries.
template <typename... P, typename... A>
cudaError_t launch_after_prep(void (*kernel)(P...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}
cudaError_t pair_capacity(int* pairs);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_quantize(const float* src, int64_t n_rows, int64_t stride,
                            const int64_t* dst_slot, uint8_t* codes, float* scales,
                            int64_t n_slots, cudaStream_t s);
cudaError_t launch_produce(const float* src, int64_t n_rows, int64_t stride, const float* weight,
                           float eps, const int64_t* positions, const float* rope_cos,
                           const float* rope_sin, int64_t max_pos, const int64_t* dst_slot,
                           uint8_t* codes, float* scales, int64_t n_slots, unsigned* err,
                           cudaStream_t s);
cudaError_t launch_prefill(const uint8_t* codes, const float* scales, const int64_t* slots,
                           int64_t n_slots, int64_t T, const uint16_t* w, int N, uint16_t* y,
                           float* k_rope, unsigned* err, cudaStream_t s);
cudaError_t launch_wait_timeout(unsigned* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_wuv(const float* o, const uint16_t* w, int B, int H, int V, float* y,
                       cudaStream_t s);

}  // namespace kv8
