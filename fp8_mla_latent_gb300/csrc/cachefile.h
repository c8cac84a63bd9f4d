// cachefile.h -- the cache file's byte layout and its host-side handling, with
// no CUDA in it (so that it also builds, with the sanitizers, in a host-only
// test): header build and parse, the open-time repair and checks, the commit of
// a row count, and the version 1 -> 2 rewrite around a caller's quantizer.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
// description, persistence item: version 2 starts with the magic COLIKV2 and
// records its data type in its header; its rows are the fp8 codes with their
// scales; a version-1 file (f32 rows) is rewritten as version 2; opening repairs
// a damaged magic.  The byte layout (the page gives none) is stated in fp8mla.h.
#pragma once
#include <errno.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

#include <string>

#include "fp8mla.h"

namespace kv8 {
namespace cachefile {

constexpr int D = 576;           // bytes of codes per row
constexpr int HDR = 64;          // header bytes
constexpr int REC2 = D + 8;      // version-2 record: codes, then sLc and sRc
constexpr int REC1 = D * 4;      // version-1 record: 576 f32
const char MAGIC2[8] = {'C', 'O', 'L', 'I', 'K', 'V', '2', 0};
const char MAGIC1[8] = {'C', 'O', 'L', 'I', 'K', 'V', '1', 0};

inline void put_u32(uint8_t* p, uint32_t v) { memcpy(p, &v, 4); }
inline void put_u64(uint8_t* p, uint64_t v) { memcpy(p, &v, 8); }
inline uint32_t get_u32(const uint8_t* p) {
  uint32_t v;
  memcpy(&v, p, 4);
  return v;
}
inline uint64_t get_u64(const uint8_t* p) {
  uint64_t v;
  memcpy(&v, p, 8);
  return v;
}

inline void make_header(uint8_t* h, int version, int64_t n_rows) {
  memset(h, 0, HDR);
  memcpy(h, version == 2 ? MAGIC2 : MAGIC1, 8);
  put_u32(h + 8, HDR);
  put_u32(h + 12, version == 2 ? 2u : 1u);
  put_u32(h + 16, D);
  put_u32(h + 20, version == 2 ? REC2 : REC1);
  put_u64(h + 24, (uint64_t)n_rows);
}

// Version of a header from its fields after the magic (0 if they fit neither).
inline int version_of_fields(const uint8_t* h) {
  if (get_u32(h + 8) != HDR || get_u32(h + 16) != D) return 0;
  if (get_u32(h + 12) == 2 && get_u32(h + 20) == REC2) return 2;
  if (get_u32(h + 12) == 1 && get_u32(h + 20) == REC1) return 1;
  return 0;
}

inline bool write_at(FILE* f, int64_t off, const void* p, size_t n) {
  if (off < 0 || fseeko(f, (off_t)off, SEEK_SET) != 0) return false;
  return n == 0 || fwrite(p, 1, n, f) == n;
}
inline bool read_at(FILE* f, int64_t off, void* p, size_t n) {
  if (off < 0 || fseeko(f, (off_t)off, SEEK_SET) != 0) return false;
  return n == 0 || fread(p, 1, n, f) == n;
}

// Write the header with this row count and flush: the commit point of an append
// (the records are written first, so a torn append is never part of the file).
inline int commit(FILE* f, int version, int64_t n_rows) {
  uint8_t h[HDR];
  make_header(h, version, n_rows);
  if (!write_at(f, 0, h, HDR) || fflush(f) != 0) return KV8_EIO;
  return KV8_OK;
}

// The header of a file just opened for reading and writing.  A file shorter than
// a header (empty, or torn at creation) becomes a fresh version-2 file of 0 rows;
// a header whose fields fit a version but whose magic is damaged is repaired; one
// whose fields fit neither version, a negative or too large row count, or a file
// with fewer bytes than its committed rows is KV8_EFORMAT.
inline int open_header(FILE* f, int* version, int64_t* n_rows) {
  uint8_t h[HDR];
  if (fseeko(f, 0, SEEK_SET) != 0) return KV8_EIO;
  const size_t got = fread(h, 1, HDR, f);
  if (got < (size_t)HDR) {
    if (ferror(f)) return KV8_EIO;
    if (ftruncate(fileno(f), 0) != 0) return KV8_EIO;
    *version = 2;
    *n_rows = 0;
    return commit(f, 2, 0);
  }
  const int v = version_of_fields(h);
  if (v == 0) return KV8_EFORMAT;
  const uint64_t rows = get_u64(h + 24);
  const uint64_t rec = v == 2 ? REC2 : REC1;
  if (rows > (uint64_t)(INT64_MAX - HDR) / rec) return KV8_EFORMAT;
  struct stat sb;
  if (fstat(fileno(f), &sb) != 0) return KV8_EIO;
  if ((uint64_t)sb.st_size < (uint64_t)HDR + rows * rec) return KV8_EFORMAT;  // rows not all there
  *version = v;
  *n_rows = (int64_t)rows;
  if (memcmp(h, v == 2 ? MAGIC2 : MAGIC1, 8) != 0) return commit(f, v, *n_rows);  // repair
  return KV8_OK;
}

// Turns the first m version-1 rows of `buf` (m * REC1 bytes of f32) into m
// version-2 records at the start of the same buffer; returns a kv8 status.
typedef int (*QuantizeRecords)(void* ctx, int64_t m, uint8_t* buf);

// Version 1 -> 2: the rows of *f are quantized chunk by chunk (chunk_rows at a
// time through buf, chunk_rows * REC1 bytes) into a new file beside `path`, which
// then replaces it; *f is reopened on the new file.  On an error the old file is
// left as it was.
inline int rewrite_v1_to_v2(const std::string& path, FILE** f, int64_t n_rows, int64_t chunk_rows,
                            uint8_t* buf, QuantizeRecords quantize, void* ctx) {
  if (chunk_rows < 1 || n_rows < 0) return KV8_EINVAL;
  const std::string tmp = path + ".v2tmp";
  FILE* g = fopen(tmp.c_str(), "w+b");
  if (g == nullptr) return KV8_EIO;
  uint8_t h[HDR];
  make_header(h, 2, 0);
  int st = fwrite(h, 1, HDR, g) == HDR ? KV8_OK : KV8_EIO;
  for (int64_t r0 = 0; st == KV8_OK && r0 < n_rows; r0 += chunk_rows) {
    const int64_t m = (n_rows - r0) < chunk_rows ? (n_rows - r0) : chunk_rows;
    if (!read_at(*f, HDR + r0 * REC1, buf, (size_t)(m * REC1))) {
      st = KV8_EIO;
      break;
    }
    st = quantize(ctx, m, buf);
    if (st == KV8_OK && fwrite(buf, 1, (size_t)(m * REC2), g) != (size_t)(m * REC2)) st = KV8_EIO;
  }
  if (st == KV8_OK) {
    make_header(h, 2, n_rows);
    if (!write_at(g, 0, h, HDR) || fflush(g) != 0 || fsync(fileno(g)) != 0) st = KV8_EIO;
  }
  if (fclose(g) != 0 && st == KV8_OK) st = KV8_EIO;
  if (st != KV8_OK) {
    remove(tmp.c_str());
    return st;
  }
  fclose(*f);
  *f = nullptr;
  if (rename(tmp.c_str(), path.c_str()) != 0) return KV8_EIO;
  *f = fopen(path.c_str(), "r+b");
  return *f != nullptr ? KV8_OK : KV8_EIO;
}

}  // namespace cachefile
}  // namespace kv8
