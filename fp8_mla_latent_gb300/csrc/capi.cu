// capi.cu -- the extern "C" boundary of libfp8mla.so: argument checks, split
// planning and kernel dispatch.  Declarations and the contract of every call
// are in include/fp8mla.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fp8mla.h"
#include "kv8_internal.h"

namespace kv8 {

static int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool tc_available();  // decode_tc.cu

SplitPlan plan_decode(int B, int H, int64_t max_len, int variant) {
  SplitPlan p{};
  int v = variant;
  if (v == kAuto) v = (H >= 16 && tc_available()) ? kTc : kSimt;
  if (v == kTc) v = (H > 64) ? kTcPair : kTcCta;
  p.variant = v;
  if (v == kTcPair) {
    p.hg = 128;  // MMA M = heads of the item, on a pair of SMs
  } else if (v == kTcCta) {
    p.hg = H <= 16 ? 16 : 32;  // heads per CTA (the MMA N is twice that: hi and lo terms)
  } else {
    p.hg = 4;
  }
  p.n_hg = (H + p.hg - 1) / p.hg;
  (void)max_len;
  // One wave: the one-CTA tensor-core kernel holds a whole SM per CTA, the pair
  // kernel two SMs per item (the launch lowers this to the pairs the device
  // holds at once), and the SIMT kernel one CTA per SM as well (its 256 threads
  // keep four tokens' rows in registers: over 200 registers each).  Cutting every
  // (sequence, head group) into items of ceil(jobs / target) tiles gives at most
  // target + B * n_hg items.
  p.target = v == kTcPair ? NUM_SMS / 2 : NUM_SMS;
  p.max_items = p.target + B * p.n_hg;
  const int64_t parts = (int64_t)p.max_items * p.hg;
  p.off_seg = 64;  // header: error word, then the item table of the split
  p.hdr_bytes = align_up(p.off_seg + (int64_t)B * p.n_hg * 16, 256);
  int64_t off = p.hdr_bytes;
  p.off_m = off;
  off = align_up(off + parts * 4, 256);
  p.off_l = off;
  off = align_up(off + parts * 4, 256);
  p.off_o = off;
  off = align_up(off + parts * DL * 4, 256);
  if (v == kTcPair || v == kTcCta) {
    p.off_q8 = off;
    off = align_up(off + (int64_t)B * H * Q8_BYTES, 256);
    p.off_cq = off;
    off = align_up(off + (int64_t)B * H * 4, 256);
  }
  p.ws_bytes = off;
  return p;
}

}  // namespace kv8

using namespace kv8;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The CUDA error behind this thread's most recent KV8_ECUDA / KV8_EUNSUPPORTED
// from a decode launch (kv8_last_cuda_error reports its name).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int bind_workspace(DecodeArgs& a, const void* workspace, int64_t workspace_bytes) {
  if (workspace == nullptr || workspace_bytes < a.plan.ws_bytes) return KV8_EWORKSPACE;
  if (!aligned(workspace, 256)) return KV8_EALIGN;
  char* ws = static_cast<char*>(const_cast<void*>(workspace));
  a.err = reinterpret_cast<unsigned*>(ws);
  a.seg = reinterpret_cast<int64_t*>(ws + a.plan.off_seg);
  a.ws_m = reinterpret_cast<float*>(ws + a.plan.off_m);
  a.ws_l = reinterpret_cast<float*>(ws + a.plan.off_l);
  a.ws_o = reinterpret_cast<float*>(ws + a.plan.off_o);
  a.q8 = a.plan.off_q8 ? reinterpret_cast<uint8_t*>(ws + a.plan.off_q8) : nullptr;
  a.cq = a.plan.off_cq ? reinterpret_cast<float*>(ws + a.plan.off_cq) : nullptr;
  return KV8_OK;
}

int run_partials(DecodeArgs& a, cudaStream_t s) {
  if (cudaMemsetAsync(a.err, 0, a.plan.hdr_bytes, s) != cudaSuccess) return KV8_ECUDA;
  cudaError_t e = a.plan.variant == kTcPair  ? launch_decode_pair(a, s)
                  : a.plan.variant == kTcCta ? launch_decode_tc(a, s)
                                             : launch_decode_simt(a, s);
  if (e != cudaSuccess) {
    g_last_cuda_error = e;
    return e == cudaErrorNotSupported ? KV8_EUNSUPPORTED : KV8_ECUDA;
  }
  return KV8_OK;
}

int run_decode(DecodeArgs& a, void* workspace, int64_t workspace_bytes, cudaStream_t s) {
  int st = bind_workspace(a, workspace, workspace_bytes);
  if (st != KV8_OK) return st;
  st = run_partials(a, s);
  if (st != KV8_OK) return st;
  const cudaError_t e = launch_combine(a, s);
  if (e != cudaSuccess) {
    g_last_cuda_error = e;
    return KV8_ECUDA;
  }
  return KV8_OK;
}

bool valid_variant(int v) { return v >= kAuto && v <= kTcPair; }

// The softmax scale: positive and finite (the kernels take running maxima of
// the raw dot products, which is only the maximum of the scores for a scale > 0).
bool valid_scale(float s) { return s > 0.0f && s <= 3.0e38f; }

}  // namespace

extern "C" {

int kv8_abi_version(void) { return 101; }

const char* kv8_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

const char* kv8_status_string(int status) {
  switch (status) {
    case KV8_OK: return "ok";
    case KV8_EINVAL: return "invalid argument";
    case KV8_EALIGN: return "pointer or stride misaligned";
    case KV8_EUNSUPPORTED: return "unsupported size or variant";
    case KV8_ECUDA: return "CUDA error";
    case KV8_EBOUNDS: return "device-side index out of range";
    case KV8_EWORKSPACE: return "workspace missing or too small";
    case KV8_ETIMEOUT: return "device-side wait timed out";
    case KV8_ESCRATCH: return "problem needs more scratch than the static no-alloc buffer";
    case KV8_EIO: return "cache file read, write or rename failed";
    case KV8_EFORMAT: return "not a cache file, or shorter than its committed rows";
    default: return "unknown status";
  }
}

int kv8_quantize_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                      const int64_t* dst_slot, uint8_t* kv_codes, float* kv_scales,
                      int64_t n_slots, void* stream) {
  if (n_rows < 0 || n_slots < 0) return KV8_EINVAL;
  if (n_rows == 0) return KV8_OK;
  if (src == nullptr || kv_codes == nullptr || kv_scales == nullptr) return KV8_EINVAL;
  if (src_row_stride < KV8_D) return KV8_EINVAL;
  if (dst_slot == nullptr && n_rows > n_slots) return KV8_EINVAL;
  if (!aligned(src, 16) || (src_row_stride % 4) != 0 || !aligned(kv_codes, 16) ||
      !aligned(kv_scales, 8))
    return KV8_EALIGN;
  cudaError_t e = launch_quantize(src, n_rows, src_row_stride, dst_slot, kv_codes, kv_scales,
                                  n_slots, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV8_OK : KV8_ECUDA;
}

int kv8_produce_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                     const float* norm_weight, float eps, const int64_t* positions,
                     const float* rope_cos, const float* rope_sin, int64_t max_pos,
                     const int64_t* dst_slot, uint8_t* kv_codes, float* kv_scales,
                     int64_t n_slots, unsigned* err_word, void* stream) {
  if (n_rows < 0 || n_slots < 0 || max_pos < 1) return KV8_EINVAL;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return KV8_EINVAL;  // also rejects NaN
  if (n_rows == 0) return KV8_OK;
  if (src == nullptr || norm_weight == nullptr || positions == nullptr || rope_cos == nullptr ||
      rope_sin == nullptr || kv_codes == nullptr || kv_scales == nullptr)
    return KV8_EINVAL;
  if (src_row_stride < KV8_D) return KV8_EINVAL;
  if (dst_slot == nullptr && n_rows > n_slots) return KV8_EINVAL;
  if (!aligned(src, 16) || (src_row_stride % 4) != 0 || !aligned(norm_weight, 16) ||
      !aligned(positions, 8) || !aligned(rope_cos, 4) || !aligned(rope_sin, 4) ||
      !aligned(kv_codes, 16) || !aligned(kv_scales, 8) || !aligned(err_word, 4))
    return KV8_EALIGN;
  cudaError_t e = launch_produce(src, n_rows, src_row_stride, norm_weight, eps, positions,
                                 rope_cos, rope_sin, max_pos, dst_slot, kv_codes, kv_scales,
                                 n_slots, err_word, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV8_OK : KV8_ECUDA;
}

int kv8_prefill_project(const uint8_t* kv_codes, const float* kv_scales, int64_t n_slots,
                        const int64_t* slots, int64_t T, const uint16_t* w_ukv, int N,
                        uint16_t* y, float* k_rope, unsigned* err_word, void* stream) {
  if (T < 0 || T > (int64_t)1 << 30 || n_slots < 0 || N < 256 || (N % 256) != 0) return KV8_EINVAL;
  if (T == 0) return KV8_OK;
  if (kv_codes == nullptr || kv_scales == nullptr || w_ukv == nullptr || y == nullptr)
    return KV8_EINVAL;
  if (slots == nullptr && T > n_slots) return KV8_EINVAL;
  if (!aligned(kv_codes, 16) || !aligned(kv_scales, 8) || !aligned(slots, 8) ||
      !aligned(w_ukv, 16) || !aligned(y, 16) || !aligned(k_rope, 16) || !aligned(err_word, 4))
    return KV8_EALIGN;
  cudaError_t e = launch_prefill(kv_codes, kv_scales, slots, n_slots, T, w_ukv, N, y, k_rope, err_word,
                                 static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return KV8_EUNSUPPORTED;
  return e == cudaSuccess ? KV8_OK : KV8_ECUDA;
}

int kv8_selftest_wait_timeout(void* workspace, int64_t workspace_bytes, int64_t limit_us,
                              void* stream) {
  if (limit_us < 1 || limit_us > 10000000) return KV8_EINVAL;
  if (workspace == nullptr || workspace_bytes < 256) return KV8_EWORKSPACE;
  if (!aligned(workspace, 256)) return KV8_EALIGN;
  unsigned* err = static_cast<unsigned*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(err, 0, sizeof(unsigned), s) != cudaSuccess) return KV8_ECUDA;
  return launch_wait_timeout(err, (uint64_t)limit_us * 1000u, s) == cudaSuccess ? KV8_OK
                                                                                : KV8_ECUDA;
}

int mla_wuv_epilogue(const float* o, const uint16_t* w_uv, int B, int H, int V, float* y,
                     void* stream) {
  if (B < 0 || H < 1 || H > 1024 || V < 1 || V > 4096) return KV8_EINVAL;
  if (B == 0) return KV8_OK;
  if (o == nullptr || w_uv == nullptr || y == nullptr) return KV8_EINVAL;
  if (!aligned(o, 4) || !aligned(w_uv, 2) || !aligned(y, 4)) return KV8_EALIGN;
  cudaError_t e = launch_wuv(o, w_uv, B, H, V, y, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV8_OK : KV8_ECUDA;
}

int64_t mla_absorb_decode_fp8_workspace_size(int64_t T, int H, int variant) {
  if (T < 0 || H < 1 || H > 1024 || !valid_variant(variant)) return -1;
  return plan_decode(1, H, T, variant).ws_bytes;
}

int mla_absorb_decode_fp8(const float* q_lat, const float* q_rope, const uint8_t* kv_codes,
                          const float* kv_scales, int64_t T, int H, float sm_scale, float* out,
                          float* lse, void* workspace, int64_t workspace_bytes, int variant,
                          void* stream) {
  if (T < 0 || H < 1 || H > 1024 || !valid_variant(variant) || !valid_scale(sm_scale))
    return KV8_EINVAL;
  if (q_lat == nullptr || q_rope == nullptr || out == nullptr) return KV8_EINVAL;
  if (T > 0 && (kv_codes == nullptr || kv_scales == nullptr)) return KV8_EINVAL;
  if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(out, 16) ||
      !aligned(kv_codes, 16) || !aligned(kv_scales, 16) || !aligned(lse, 4))
    return KV8_EALIGN;
  DecodeArgs a{};
  a.q_lat = q_lat;
  a.q_rope = q_rope;
  a.codes = kv_codes;
  a.scales = kv_scales;
  a.block_table = nullptr;
  a.seq_lens = nullptr;
  a.T_contig = T;
  a.B = 1;
  a.H = H;
  a.max_blocks = 0;
  a.n_blocks = 0;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.plan = plan_decode(1, H, T, variant);
  return run_decode(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int64_t mla_absorb_decode_fp8_batch_workspace_size(int B, int H, int max_blocks, int block_size,
                                                   int variant) {
  if (B < 0 || H < 1 || H > 1024 || max_blocks < 1 || block_size != KV8_BLOCK ||
      !valid_variant(variant))
    return -1;
  return plan_decode(B, H, (int64_t)max_blocks * block_size, variant).ws_bytes;
}

}  // extern "C"

namespace {

int batch_args(DecodeArgs& a, const float* q_lat, const float* q_rope, const uint8_t* kv_codes,
               const float* kv_scales, const int32_t* block_table, const int32_t* seq_lens,
               int B, int H, int max_blocks, int block_size, int64_t n_blocks, float sm_scale,
               float* out, float* lse, int variant, bool need_inputs, bool need_outputs) {
  if (B < 0 || H < 1 || H > 1024 || max_blocks < 1 || !valid_variant(variant)) return KV8_EINVAL;
  if (need_inputs && (n_blocks < 1 || !valid_scale(sm_scale))) return KV8_EINVAL;
  if (block_size != KV8_BLOCK) return KV8_EUNSUPPORTED;
  if (seq_lens == nullptr || !aligned(seq_lens, 4)) return seq_lens ? KV8_EALIGN : KV8_EINVAL;
  if (need_inputs) {
    if (q_lat == nullptr || q_rope == nullptr || kv_codes == nullptr || kv_scales == nullptr ||
        block_table == nullptr)
      return KV8_EINVAL;
    if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(kv_codes, 16) ||
        !aligned(kv_scales, 16) || !aligned(block_table, 4))
      return KV8_EALIGN;
  }
  if (need_outputs) {
    if (out == nullptr) return KV8_EINVAL;
    if (!aligned(out, 16) || !aligned(lse, 4)) return KV8_EALIGN;
  }
  a = DecodeArgs{};
  a.q_lat = q_lat;
  a.q_rope = q_rope;
  a.codes = kv_codes;
  a.scales = kv_scales;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.T_contig = 0;
  a.B = B;
  a.H = H;
  a.max_blocks = max_blocks;
  a.n_blocks = n_blocks;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.plan = plan_decode(B, H, (int64_t)max_blocks * block_size, variant);
  return KV8_OK;
}

}  // namespace

extern "C" {

int mla_absorb_decode_fp8_batch(const float* q_lat, const float* q_rope, const uint8_t* kv_codes,
                                const float* kv_scales, const int32_t* block_table,
                                const int32_t* seq_lens, int B, int H, int max_blocks,
                                int block_size, int64_t n_blocks, float sm_scale, float* out,
                                float* lse, void* workspace, int64_t workspace_bytes,
                                int variant, void* stream) {
  DecodeArgs a;
  int st = batch_args(a, q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, B, H,
                      max_blocks, block_size, n_blocks, sm_scale, out, lse, variant, true, true);
  if (st != KV8_OK || B == 0) return st;
  return run_decode(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int mla_absorb_decode_fp8_batch_partials(const float* q_lat, const float* q_rope,
                                         const uint8_t* kv_codes, const float* kv_scales,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int B, int H, int max_blocks, int block_size,
                                         int64_t n_blocks, float sm_scale, void* workspace,
                                         int64_t workspace_bytes, int variant, void* stream) {
  DecodeArgs a;
  int st = batch_args(a, q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, B, H,
                      max_blocks, block_size, n_blocks, sm_scale, nullptr, nullptr, variant, true,
                      false);
  if (st != KV8_OK || B == 0) return st;
  st = bind_workspace(a, workspace, workspace_bytes);
  if (st != KV8_OK) return st;
  return run_partials(a, static_cast<cudaStream_t>(stream));
}

int mla_absorb_decode_fp8_batch_combine(const int32_t* seq_lens, int B, int H, int max_blocks,
                                        int block_size, float* out, float* lse,
                                        const void* workspace, int64_t workspace_bytes,
                                        int variant, void* stream) {
  DecodeArgs a;
  int st = batch_args(a, nullptr, nullptr, nullptr, nullptr, nullptr, seq_lens, B, H,
                      max_blocks, block_size, 0, 0.f, out, lse, variant, false, true);
  if (st != KV8_OK || B == 0) return st;
  st = bind_workspace(a, workspace, workspace_bytes);
  if (st != KV8_OK) return st;
  const cudaError_t e = launch_combine(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) g_last_cuda_error = e;
  return e == cudaSuccess ? KV8_OK : KV8_ECUDA;
}

int kv8_workspace_error(const void* workspace, void* stream) {
  if (workspace == nullptr) return KV8_EINVAL;
  unsigned w = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&w, workspace, sizeof w, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KV8_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KV8_ECUDA;
  if (w & ERR_TIMEOUT) return KV8_ETIMEOUT;
  return w ? KV8_EBOUNDS : KV8_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation decode.  For callers that cannot allocate device memory (a host
// runtime that owns every buffer and passes only inputs and outputs, or a loop
// with a fixed memory budget): the split-T partials live in one scratch array
// declared here, in device memory, for the life of the process.  In host code
// the array's name is only a stand-in for the symbol, never a device address:
// its address is looked up once per device with cudaGetSymbolAddress.

namespace {

constexpr int64_t kNoallocBytes = KV8_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up on first use).
int noalloc_scratch(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV8_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return KV8_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return KV8_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return KV8_OK;
}

}  // namespace

extern "C" {

int mla_absorb_decode_fp8_batch_noalloc(const float* q_lat, const float* q_rope,
                                        const uint8_t* kv_codes, const float* kv_scales,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int B, int H, int max_blocks, int block_size,
                                        int64_t n_blocks, float sm_scale, float* out,
                                        float* lse, int variant, void* stream) {
  DecodeArgs a;
  int st = batch_args(a, q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, B, H,
                      max_blocks, block_size, n_blocks, sm_scale, out, lse, variant, true, true);
  if (st != KV8_OK || B == 0) return st;
  if (a.plan.ws_bytes > kNoallocBytes) return KV8_ESCRATCH;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != KV8_OK) return st;
  // run_decode clears the error word before the split kernel; the partials are
  // written before they are read, so nothing else needs zeroing.
  return run_decode(a, scratch, kNoallocBytes, static_cast<cudaStream_t>(stream));
}

int kv8_noalloc_error(void* stream) {
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != KV8_OK) return st;
  return kv8_workspace_error(scratch, stream);
}

}  // extern "C"
