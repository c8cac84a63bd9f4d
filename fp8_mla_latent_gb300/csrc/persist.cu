// persist.cu -- save and resume of the fp8 cache through a cache file.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
// description, persistence item: version 2 of the cache file starts with the
// magic COLIKV2 and records its data type in its header; its rows are the fp8
// codes with their scales; rows are appended through a persistent handle with a
// staging buffer; a version-1 file (f32 rows) is quantized on resume and
// rewritten as version 2 at the first append; opening repairs a damaged magic.
// The byte layout (the page gives none) is stated in fp8mla.h.
//
// A handle owns the open file and a pinned, device-mapped host staging buffer.
// Append: a gather kernel packs the rows of the requested cache slots into
// 584-byte records straight into the staging buffer (over the host link), the
// host writes them after the last committed record, and only then rewrites the
// header's row count, so a torn append is never part of the file.  Load: the
// host reads records into the staging buffer and a scatter kernel puts them into
// cache slots; version-1 rows go through the library's quantizer instead.  The
// records use two buffers, so the kernel of one chunk overlaps the file transfer
// of the next (append) or previous (load).
#include <errno.h>
#include <stdio.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

#include <string>

#include "cachefile.h"
#include "fp8mla.h"
#include "kv8_internal.h"

namespace kv8 {
namespace {

using cachefile::HDR;
using cachefile::read_at;
using cachefile::REC1;
using cachefile::REC2;
using cachefile::write_at;
constexpr int STAGE_ROW = REC1 + D + 8;  // f32 rows (or records) + codes + scales per staged row

// One warp per record; a record is 73 eight-byte words (72 of codes, 1 of scales).
__global__ void gather_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                              int64_t n_slots, const int64_t* __restrict__ slots, int64_t first,
                              int64_t n, uint8_t* __restrict__ rec, int* flag) {
  const int lane = threadIdx.x & 31;
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (i >= n) return;
  const int64_t slot = slots != nullptr ? slots[i] : first + i;
  uint64_t* dst = reinterpret_cast<uint64_t*>(rec + i * REC2);
  if (slot < 0 || slot >= n_slots) {
    for (int k = lane; k < REC2 / 8; k += 32) dst[k] = 0;
    if (lane == 0) *reinterpret_cast<volatile int*>(flag) = 1;
    return;
  }
  const uint64_t* src = reinterpret_cast<const uint64_t*>(codes + slot * D);
  for (int k = lane; k < D / 8; k += 32) dst[k] = src[k];
  if (lane == 0) dst[D / 8] = *reinterpret_cast<const uint64_t*>(scales + slot * 2);
}

__global__ void scatter_kernel(const uint8_t* __restrict__ rec, int64_t n, uint8_t* __restrict__ codes,
                               float* __restrict__ scales, int64_t n_slots,
                               const int64_t* __restrict__ slots, int64_t first, int* flag) {
  const int lane = threadIdx.x & 31;
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (i >= n) return;
  const int64_t slot = slots != nullptr ? slots[i] : first + i;
  if (slot < 0 || slot >= n_slots) {
    if (lane == 0) *reinterpret_cast<volatile int*>(flag) = 1;
    return;
  }
  const uint64_t* src = reinterpret_cast<const uint64_t*>(rec + i * REC2);
  uint64_t* dst = reinterpret_cast<uint64_t*>(codes + slot * D);
  for (int k = lane; k < D / 8; k += 32) dst[k] = src[k];
  if (lane == 0) *reinterpret_cast<uint64_t*>(scales + slot * 2) = src[D / 8];
}

__global__ void check_slots_kernel(const int64_t* __restrict__ slots, int64_t n, int64_t n_slots,
                                   int* flag) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && (slots[i] < 0 || slots[i] >= n_slots)) *reinterpret_cast<volatile int*>(flag) = 1;
}

}  // namespace
}  // namespace kv8

using namespace kv8;

struct kv8_disk {
  FILE* f = nullptr;
  std::string path;
  int version = 2;
  int64_t n_rows = 0;
  int64_t staging_rows = 0;
  uint8_t* stage = nullptr;   // pinned, mapped: staging_rows x STAGE_ROW bytes
  uint8_t* stage_dev = nullptr;
  int* flag = nullptr;        // pinned, mapped: set by the kernels on a bad slot
  int* flag_dev = nullptr;
};

namespace {

// the three areas of the staging buffer (host and device views)
uint8_t* area_rows(kv8_disk* d, bool dev) { return dev ? d->stage_dev : d->stage; }
uint8_t* area_codes(kv8_disk* d, bool dev) {
  return (dev ? d->stage_dev : d->stage) + d->staging_rows * REC1;
}
float* area_scales(kv8_disk* d, bool dev) {
  return reinterpret_cast<float*>((dev ? d->stage_dev : d->stage) + d->staging_rows * (REC1 + D));
}

int commit_rows(kv8_disk* d, int64_t n_rows) {
  const int st = cachefile::commit(d->f, d->version, n_rows);
  if (st == KV8_OK) d->n_rows = n_rows;
  return st;
}

// Version 1 -> 2: the file's rewrite (cachefile.h) with the library's quantizer:
// the staged f32 rows through the device view of the staging buffer, then codes
// and scales interleaved into records over the (now free) f32 area.
struct ConvertCtx {
  kv8_disk* d;
  cudaStream_t s;
};
int quantize_records(void* ctx, int64_t m, uint8_t* buf) {
  kv8_disk* d = static_cast<ConvertCtx*>(ctx)->d;
  cudaStream_t s = static_cast<ConvertCtx*>(ctx)->s;
  if (buf != area_rows(d, false)) return KV8_EINVAL;
  if (launch_quantize(reinterpret_cast<const float*>(area_rows(d, true)), m, D, nullptr,
                      area_codes(d, true), area_scales(d, true), m, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return KV8_ECUDA;
  const uint8_t* c = area_codes(d, false);
  const float* sc = area_scales(d, false);
  for (int64_t i = 0; i < m; ++i) {
    memcpy(buf + i * REC2, c + i * D, D);
    memcpy(buf + i * REC2 + D, sc + i * 2, 8);
  }
  return KV8_OK;
}
int convert_to_v2(kv8_disk* d, cudaStream_t s) {
  ConvertCtx ctx{d, s};
  const int st = cachefile::rewrite_v1_to_v2(d->path, &d->f, d->n_rows, d->staging_rows,
                                             area_rows(d, false), quantize_records, &ctx);
  if (st == KV8_OK) d->version = 2;
  return st;
}

}  // namespace

extern "C" {

int kv8_disk_open(const char* path, int64_t staging_rows, kv8_disk** out) {
  if (out == nullptr) return KV8_EINVAL;
  *out = nullptr;
  if (path == nullptr || path[0] == 0 || staging_rows < 1 || staging_rows > (int64_t)1 << 22)
    return KV8_EINVAL;
  kv8_disk* d = new kv8_disk();
  d->path = path;
  d->staging_rows = staging_rows;
  void* p = nullptr;
  if (cudaHostAlloc(&p, (size_t)(staging_rows * STAGE_ROW) + 64, cudaHostAllocMapped) != cudaSuccess) {
    delete d;
    return KV8_ECUDA;
  }
  d->stage = static_cast<uint8_t*>(p);
  d->flag = reinterpret_cast<int*>(d->stage + staging_rows * STAGE_ROW);
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, p, 0) != cudaSuccess) {
    cudaFreeHost(p);
    delete d;
    return KV8_ECUDA;
  }
  d->stage_dev = static_cast<uint8_t*>(dp);
  d->flag_dev = reinterpret_cast<int*>(d->stage_dev + staging_rows * STAGE_ROW);

  int st = KV8_OK;
  d->f = fopen(path, "r+b");
  if (d->f == nullptr && errno == ENOENT) d->f = fopen(path, "w+b");
  if (d->f == nullptr) st = KV8_EIO;
  if (st == KV8_OK) st = cachefile::open_header(d->f, &d->version, &d->n_rows);
  if (st != KV8_OK) {
    kv8_disk_close(d);
    return st;
  }
  *out = d;
  return KV8_OK;
}

int kv8_disk_info(const kv8_disk* d, int64_t* n_rows, int* version) {
  if (d == nullptr) return KV8_EINVAL;
  if (n_rows != nullptr) *n_rows = d->n_rows;
  if (version != nullptr) *version = d->version;
  return KV8_OK;
}

int kv8_disk_append(kv8_disk* d, const uint8_t* kv_codes, const float* kv_scales, int64_t n_slots,
                    const int64_t* slots, int64_t n, void* stream) {
  if (d == nullptr || n < 0 || n_slots < 0) return KV8_EINVAL;
  if (n == 0) return KV8_OK;
  if (kv_codes == nullptr || kv_scales == nullptr) return KV8_EINVAL;
  if (slots == nullptr && n > n_slots) return KV8_EINVAL;
  if (((uintptr_t)kv_codes & 15) || ((uintptr_t)kv_scales & 7) || ((uintptr_t)slots & 7))
    return KV8_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->version == 1) {
    const int st = convert_to_v2(d, s);
    if (st != KV8_OK) return st;
  }
  // two record buffers in the staging area: the gather of chunk k + 1 runs on the
  // device while the host writes chunk k
  const int64_t cap = d->staging_rows;
  auto launch = [&](int64_t r0, int b) -> bool {
    const int64_t m = (n - r0) < cap ? (n - r0) : cap;
    *reinterpret_cast<volatile int*>(d->flag) = 0;
    gather_kernel<<<(unsigned)((m * 32 + 255) / 256), 256, 0, s>>>(
        kv_codes, kv_scales, n_slots, slots != nullptr ? slots + r0 : nullptr, r0, m,
        area_rows(d, true) + b * cap * REC2, d->flag_dev);
    return cudaGetLastError() == cudaSuccess;
  };
  if (!launch(0, 0)) return KV8_ECUDA;
  for (int64_t r0 = 0, k = 0; r0 < n; r0 += cap, ++k) {
    const int64_t m = (n - r0) < cap ? (n - r0) : cap;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV8_ECUDA;
    if (*reinterpret_cast<volatile int*>(d->flag) != 0) return KV8_EBOUNDS;  // nothing committed
    if (r0 + cap < n && !launch(r0 + cap, (int)((k + 1) & 1))) return KV8_ECUDA;
    if (!write_at(d->f, HDR + (d->n_rows + r0) * REC2, area_rows(d, false) + (k & 1) * cap * REC2,
                  (size_t)(m * REC2))) {
      cudaStreamSynchronize(s);
      return KV8_EIO;
    }
  }
  if (fflush(d->f) != 0) return KV8_EIO;
  return commit_rows(d, d->n_rows + n);
}

int kv8_disk_load(kv8_disk* d, int64_t first_row, int64_t n, uint8_t* kv_codes, float* kv_scales,
                  int64_t n_slots, const int64_t* dst_slot, void* stream) {
  if (d == nullptr || n < 0 || first_row < 0 || n_slots < 0) return KV8_EINVAL;
  if (first_row + n > d->n_rows) return KV8_EINVAL;
  if (n == 0) return KV8_OK;
  if (kv_codes == nullptr || kv_scales == nullptr) return KV8_EINVAL;
  if (dst_slot == nullptr && first_row + n > n_slots) return KV8_EINVAL;
  if (((uintptr_t)kv_codes & 15) || ((uintptr_t)kv_scales & 7) || ((uintptr_t)dst_slot & 7))
    return KV8_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t cap = d->staging_rows;
  if (d->version == 2) {
    // two record buffers: the host reads chunk k + 1 while the device scatters chunk k
    auto read_chunk = [&](int64_t r0, int b) -> bool {
      const int64_t m = (n - r0) < cap ? (n - r0) : cap;
      return read_at(d->f, HDR + (first_row + r0) * REC2, area_rows(d, false) + b * cap * REC2,
                     (size_t)(m * REC2));
    };
    if (!read_chunk(0, 0)) return KV8_EIO;
    *reinterpret_cast<volatile int*>(d->flag) = 0;
    for (int64_t r0 = 0, k = 0; r0 < n; r0 += cap, ++k) {
      const int64_t m = (n - r0) < cap ? (n - r0) : cap;
      scatter_kernel<<<(unsigned)((m * 32 + 255) / 256), 256, 0, s>>>(
          area_rows(d, true) + (k & 1) * cap * REC2, m, kv_codes, kv_scales, n_slots,
          dst_slot != nullptr ? dst_slot + r0 : nullptr, first_row + r0, d->flag_dev);
      if (cudaGetLastError() != cudaSuccess) return KV8_ECUDA;
      const bool more = r0 + cap < n;
      const bool read_ok = !more || read_chunk(r0 + cap, (int)((k + 1) & 1));
      if (cudaStreamSynchronize(s) != cudaSuccess) return KV8_ECUDA;
      if (!read_ok) return KV8_EIO;
    }
    return *reinterpret_cast<volatile int*>(d->flag) != 0 ? KV8_EBOUNDS : KV8_OK;
  }
  for (int64_t r0 = 0; r0 < n; r0 += cap) {
    const int64_t m = (n - r0) < cap ? (n - r0) : cap;
    const int64_t row = first_row + r0;
    const int64_t* sl = dst_slot != nullptr ? dst_slot + r0 : nullptr;
    *reinterpret_cast<volatile int*>(d->flag) = 0;
    if (!read_at(d->f, HDR + row * REC1, area_rows(d, false), (size_t)(m * REC1))) return KV8_EIO;
    // version 1: the rows are quantized on the way in (identity slots start at `row`;
    // the quantizer skips a slot outside the pool, which the check reports)
    if (sl != nullptr) {
      check_slots_kernel<<<(unsigned)((m + 255) / 256), 256, 0, s>>>(sl, m, n_slots, d->flag_dev);
      if (cudaGetLastError() != cudaSuccess) return KV8_ECUDA;
    }
    const cudaError_t e =
        sl != nullptr
            ? launch_quantize(reinterpret_cast<const float*>(area_rows(d, true)), m, D, sl,
                              kv_codes, kv_scales, n_slots, s)
            : launch_quantize(reinterpret_cast<const float*>(area_rows(d, true)), m, D, nullptr,
                              kv_codes + row * D, kv_scales + row * 2, n_slots - row, s);
    if (e != cudaSuccess) return KV8_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV8_ECUDA;
    if (*reinterpret_cast<volatile int*>(d->flag) != 0) return KV8_EBOUNDS;
  }
  return KV8_OK;
}

int kv8_disk_close(kv8_disk* d) {
  if (d == nullptr) return KV8_OK;
  int st = KV8_OK;
  if (d->f != nullptr && fclose(d->f) != 0) st = KV8_EIO;
  if (d->stage != nullptr) cudaFreeHost(d->stage);
  delete d;
  return st;
}

}  // extern "C"
