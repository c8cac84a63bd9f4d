// Host-only driver run under AddressSanitizer and UndefinedBehaviorSanitizer by
// tests/test_host_sanitizers.py.  Two independent parts, each exercising host C/C++
// that takes untrusted or edge-case input:
//   1. the cache file's host code (fp8_mla_latent_gb300/csrc/cachefile.h): header
//      parse, the open-time repair of a damaged magic, torn and truncated files,
//      inconsistent headers, random headers, and the version 1 -> 2 rewrite (with
//      a stand-in row-to-record function: the file code, not the quantizer, is
//      under test here);
//   2. the oracle's C (oracle/kv8_oracle.c): every entry point on small inputs,
//      special values included.
// Exits 0 when every check holds; the sanitizers abort on the first report.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include <string>
#include <vector>

#include "cachefile.h"
#include "kv8_oracle.h"

namespace cf = kv8::cachefile;

static int failures = 0;
#define CHECK(cond)                                                        \
  do {                                                                     \
    if (!(cond)) {                                                         \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond);  \
      ++failures;                                                          \
    }                                                                      \
  } while (0)

static std::string dir;

static FILE* reopen(const std::string& path) { return fopen(path.c_str(), "r+b"); }

static long file_size(const std::string& path) {
  FILE* f = fopen(path.c_str(), "rb");
  if (!f) return -1;
  fseek(f, 0, SEEK_END);
  const long n = ftell(f);
  fclose(f);
  return n;
}

// stand-in for the quantizer: record r = the low byte of each f32 of row r, then
// the row's first two floats as its "scales"
static int fake_records(void* ctx, int64_t m, uint8_t* buf) {
  int* calls = static_cast<int*>(ctx);
  if (calls[1] > 0 && calls[0] + 1 == calls[1]) return KV8_EIO;  // planted failure at chunk calls[1]
  ++calls[0];
  std::vector<uint8_t> rec((size_t)m * cf::REC2);
  for (int64_t r = 0; r < m; ++r) {
    const float* x = reinterpret_cast<const float*>(buf + r * cf::REC1);
    for (int i = 0; i < cf::D; ++i) {
      uint32_t b;
      memcpy(&b, &x[i], 4);
      rec[r * cf::REC2 + i] = (uint8_t)(b & 0xFFu);
    }
    memcpy(&rec[r * cf::REC2 + cf::D], x, 8);
  }
  memcpy(buf, rec.data(), rec.size());
  return KV8_OK;
}

static void write_v1(const std::string& path, int64_t n) {
  FILE* f = fopen(path.c_str(), "w+b");
  uint8_t h[cf::HDR];
  cf::make_header(h, 1, n);
  fwrite(h, 1, cf::HDR, f);
  for (int64_t r = 0; r < n; ++r)
    for (int i = 0; i < cf::D; ++i) {
      const float v = (float)(r * 1000 + i) * 0.5f;
      fwrite(&v, 4, 1, f);
    }
  fclose(f);
}

static void cache_file_cases() {
  const std::string path = dir + "/a.kv";
  int version = -1;
  int64_t rows = -1;
  // a new, empty file becomes a version-2 file of 0 rows
  FILE* f = fopen(path.c_str(), "w+b");
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 2 && rows == 0);
  fclose(f);
  CHECK(file_size(path) == cf::HDR);
  // records, then the commit; the count is read back
  f = reopen(path);
  std::vector<uint8_t> rec(5 * cf::REC2);
  for (size_t i = 0; i < rec.size(); ++i) rec[i] = (uint8_t)(i * 7);
  CHECK(cf::write_at(f, cf::HDR, rec.data(), rec.size()));
  CHECK(cf::commit(f, 2, 5) == KV8_OK);
  fclose(f);
  f = reopen(path);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 2 && rows == 5);
  std::vector<uint8_t> back(rec.size());
  CHECK(cf::read_at(f, cf::HDR, back.data(), back.size()) && back == rec);
  // a damaged magic is repaired, the rows kept
  const uint8_t bad = 'X';
  CHECK(cf::write_at(f, 3, &bad, 1));
  fclose(f);
  f = reopen(path);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && rows == 5);
  uint8_t h[cf::HDR];
  CHECK(cf::read_at(f, 0, h, cf::HDR) && memcmp(h, cf::MAGIC2, 8) == 0);
  // a row count past the file's bytes, or absurdly large, is a format error
  CHECK(cf::commit(f, 2, 6) == KV8_OK);
  CHECK(cf::open_header(f, &version, &rows) == KV8_EFORMAT);
  cf::put_u64(h + 24, ~0ull);
  CHECK(cf::write_at(f, 0, h, cf::HDR));
  CHECK(cf::open_header(f, &version, &rows) == KV8_EFORMAT);
  cf::put_u64(h + 24, 1ull << 62);
  CHECK(cf::write_at(f, 0, h, cf::HDR));
  CHECK(cf::open_header(f, &version, &rows) == KV8_EFORMAT);
  // fields that fit no version
  cf::make_header(h, 2, 0);
  cf::put_u32(h + 8, 99);
  CHECK(cf::write_at(f, 0, h, cf::HDR));
  CHECK(cf::open_header(f, &version, &rows) == KV8_EFORMAT);
  cf::make_header(h, 2, 0);
  cf::put_u32(h + 20, cf::REC1);
  CHECK(cf::write_at(f, 0, h, cf::HDR));
  CHECK(cf::open_header(f, &version, &rows) == KV8_EFORMAT);
  fclose(f);
  // a file torn inside its header becomes a fresh, empty version-2 file
  CHECK(truncate(path.c_str(), 10) == 0);
  f = reopen(path);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 2 && rows == 0);
  fclose(f);
  CHECK(file_size(path) == cf::HDR);

  // version 1 -> 2, in chunks of 3 rows (7 rows: a short last chunk)
  const std::string p1 = dir + "/v1.kv";
  write_v1(p1, 7);
  f = reopen(p1);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 1 && rows == 7);
  std::vector<uint8_t> buf(3 * cf::REC1);
  int calls[2] = {0, 0};
  CHECK(cf::rewrite_v1_to_v2(p1, &f, rows, 3, buf.data(), fake_records, calls) == KV8_OK);
  CHECK(calls[0] == 3 && f != nullptr);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 2 && rows == 7);
  for (int64_t r = 0; r < 7; ++r) {
    uint8_t got[cf::REC2];
    CHECK(cf::read_at(f, cf::HDR + r * cf::REC2, got, cf::REC2));
    for (int i = 0; i < cf::D; ++i) {
      const float v = (float)(r * 1000 + i) * 0.5f;
      uint32_t b;
      memcpy(&b, &v, 4);
      if (got[i] != (uint8_t)(b & 0xFFu)) {
        CHECK(false);
        break;
      }
    }
  }
  fclose(f);
  CHECK(access((p1 + ".v2tmp").c_str(), F_OK) != 0);
  // a failing chunk leaves the version-1 file as it was and no temporary behind
  write_v1(p1, 7);
  const long before = file_size(p1);
  f = reopen(p1);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 1);
  int fail_calls[2] = {0, 2};
  CHECK(cf::rewrite_v1_to_v2(p1, &f, rows, 3, buf.data(), fake_records, fail_calls) == KV8_EIO);
  CHECK(f != nullptr && file_size(p1) == before);
  CHECK(cf::open_header(f, &version, &rows) == KV8_OK && version == 1 && rows == 7);
  fclose(f);
  CHECK(access((p1 + ".v2tmp").c_str(), F_OK) != 0);
  // bad arguments
  f = reopen(p1);
  CHECK(cf::rewrite_v1_to_v2(p1, &f, 7, 0, buf.data(), fake_records, calls) == KV8_EINVAL);
  fclose(f);

  // random headers and lengths: a status, never a crash
  const std::string pr = dir + "/r.kv";
  uint64_t s = 0x9E3779B97F4A7C15ull;
  auto next = [&]() {
    s ^= s << 13;
    s ^= s >> 7;
    s ^= s << 17;
    return s;
  };
  for (int k = 0; k < 3000; ++k) {
    FILE* g = fopen(pr.c_str(), "w+b");
    const int len = (int)(next() % 200);
    std::vector<uint8_t> bytes(len);
    for (auto& x : bytes) x = (uint8_t)next();
    if (len >= cf::HDR && (next() & 1)) {  // often a plausible header with random fields
      cf::make_header(bytes.data(), (next() & 1) ? 2 : 1, (int64_t)(next() % 4));
      bytes[next() % cf::HDR] ^= (uint8_t)(1u << (next() % 8));
    }
    if (len) fwrite(bytes.data(), 1, bytes.size(), g);
    fflush(g);
    const int st = cf::open_header(g, &version, &rows);
    CHECK(st == KV8_OK || st == KV8_EFORMAT);
    if (st == KV8_OK) CHECK((version == 1 || version == 2) && rows >= 0);
    fclose(g);
  }
}

static void oracle_cases() {
  // codec
  float lut[256];
  orc_e4m3_decode_table(lut);
  for (int c = 0; c < 256; ++c) {
    const float v = orc_e4m3_decode((uint8_t)c);
    CHECK((isnan(v) && isnan(lut[c])) || v == lut[c]);
  }
  const float specials[] = {0.f, -0.f, 448.f, -448.f, 449.f, 1e30f, -1e30f, 1e-45f, NAN, INFINITY,
                            -INFINITY, 0.0009765625f, 240.f, 232.f, 17.f};
  for (float q : specials) {
    const uint8_t a = orc_e4m3_encode(q), b = orc_e4m3_encode_nearest(q), c = orc_e4m3_encode_bracket(q);
    CHECK(a == b && a == c);
  }
  uint32_t first_bad = 0;
  CHECK(orc_e4m3_exhaustive_mismatches(0x3F000000u, 0x3F000000u + 4096u, &first_bad) == 0);
  std::vector<uint32_t> bits(256);
  for (int i = 0; i < 256; ++i) bits[i] = 0x43000000u + (uint32_t)i * 977u;
  CHECK(orc_e4m3_list_mismatches_nearest(bits.data(), 256, &first_bad) == 0);
  std::vector<float> xs(64);
  for (int i = 0; i < 64; ++i) xs[i] = (float)(i - 32) * 7.25f;
  std::vector<uint8_t> enc(64);
  for (int which = 0; which < 3; ++which) orc_e4m3_encode_array(xs.data(), 64, enc.data(), which);

  // quantizer: ordinary, zero, NaN-bearing, subnormal-amax and huge rows, through a
  // slot map with a stride wider than a row
  const int n = 8, stride = 600, n_slots = 16;
  std::vector<float> rows((size_t)n * stride, 0.f);
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < 576; ++i) rows[(size_t)r * stride + i] = sinf((float)(r * 577 + i)) * 3.f;
  for (int i = 0; i < 576; ++i) rows[1 * stride + i] = 0.f;
  rows[2 * stride + 5] = NAN;
  for (int i = 0; i < 576; ++i) rows[3 * stride + i] = 1e-42f;
  for (int i = 0; i < 576; ++i) rows[4 * stride + i] = 3e38f;
  std::vector<int64_t> slot = {15, 0, 7, 3, 9, 1, 2, 14};
  std::vector<uint8_t> codes((size_t)n_slots * 576, 0xAB);
  std::vector<float> scales((size_t)n_slots * 2, -1.f);
  orc_quantize_rows(rows.data(), n, stride, slot.data(), codes.data(), scales.data());
  orc_quantize_rows(rows.data(), n, stride, nullptr, codes.data(), scales.data());
  uint8_t c1[576];
  float s1[2];
  orc_quantize_row(rows.data(), c1, s1);
  CHECK(memcmp(c1, &codes[0], 576) == 0);

  // fused producer: norm, rotation, quantizer, positions in and out of range
  std::vector<float> w(512), ys(576), cosr(32 * 32), sinr(32 * 32);
  for (int i = 0; i < 512; ++i) w[i] = 1.f + 0.01f * (float)(i % 7);
  for (int p = 0; p < 32; ++p)
    for (int j = 0; j < 32; ++j) {
      cosr[p * 32 + j] = cosf((float)(p * (j + 1)) * 0.01f);
      sinr[p * 32 + j] = sinf((float)(p * (j + 1)) * 0.01f);
    }
  orc_rmsnorm_row(rows.data(), w.data(), 1e-6f, ys.data());
  orc_rope_pairs(rows.data() + 512, cosr.data(), sinr.data(), ys.data() + 512);
  std::vector<int64_t> pos = {0, 31, -1, 32, 5, 1ll << 40, 7, 8};
  orc_produce_rows(rows.data(), n, stride, w.data(), 1e-6f, pos.data(), cosr.data(), sinr.data(), 32,
                   slot.data(), codes.data(), scales.data());

  // attention: single sequence (f32, f64, a head range, partials and their merge) and
  // a paged batch of two sequences
  const int H = 4, T = 130;
  std::vector<float> crows((size_t)T * 576);
  for (size_t i = 0; i < crows.size(); ++i) crows[i] = cosf((float)i * 0.37f) * 2.f;
  std::vector<uint8_t> kc((size_t)T * 576);
  std::vector<float> ks((size_t)T * 2);
  orc_quantize_rows(crows.data(), T, 576, nullptr, kc.data(), ks.data());
  std::vector<float> ql((size_t)2 * H * 512), qr((size_t)2 * H * 64);
  for (size_t i = 0; i < ql.size(); ++i) ql[i] = sinf((float)i * 0.11f);
  for (size_t i = 0; i < qr.size(); ++i) qr[i] = cosf((float)i * 0.13f);
  std::vector<float> out((size_t)2 * H * 512), lse(2 * H);
  std::vector<double> out64((size_t)H * 512), lse64(H), o2((size_t)2 * H * 512), m2(2 * H), l2(2 * H);
  orc_attention_f32(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, T, H, 0.072f, out.data(), lse.data());
  orc_attention_f64(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, T, H, 0.072, out64.data(), lse64.data());
  orc_attention_heads_f64(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, T, H, 1, 2, 0.072,
                          out64.data(), lse64.data());
  orc_attention_partial_f64(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, 0, 64, H, 0.072,
                            o2.data(), m2.data(), l2.data());
  orc_attention_partial_f64(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, 64, T, H, 0.072,
                            o2.data() + (size_t)H * 512, m2.data() + H, l2.data() + H);
  orc_lse_merge_f64(2, H, o2.data(), m2.data(), l2.data(), out64.data(), lse64.data());
  orc_attention_f32(ql.data(), qr.data(), kc.data(), ks.data(), nullptr, 0, H, 0.072f, out.data(), lse.data());
  for (int i = 0; i < H * 512; ++i) CHECK(isfinite(out64[i]));
  // paged: pages of 64 tokens, sequence 0 = 130 tokens (3 pages), 1 = 1 token
  const int max_blocks = 3;
  std::vector<int32_t> bt = {2, 0, 1, 1, 0, 0};
  std::vector<int32_t> lens = {130, 1};
  std::vector<uint8_t> pc((size_t)3 * 64 * 576, 0);
  std::vector<float> ps((size_t)3 * 64 * 2, 1.f);
  std::vector<int64_t> sl(130);
  orc_paged_slots(bt.data(), max_blocks, 64, 0, 130, sl.data());
  for (int t = 0; t < 130; ++t) {
    memcpy(&pc[(size_t)sl[t] * 576], &kc[(size_t)t * 576], 576);
    memcpy(&ps[(size_t)sl[t] * 2], &ks[(size_t)t * 2], 8);
  }
  orc_attention_batch_f32(ql.data(), qr.data(), pc.data(), ps.data(), bt.data(), lens.data(), 2, H,
                          max_blocks, 64, 0.072f, out.data(), lse.data(), 2);
  for (int i = 0; i < 2 * H * 512; ++i) CHECK(isfinite(out[i]));
  CHECK(orc_max_threads() >= 1);
}

int main(int argc, char** argv) {
  dir = argc > 1 ? argv[1] : "/tmp";
  cache_file_cases();
  oracle_cases();
  if (failures) {
    fprintf(stderr, "%d checks failed\n", failures);
    return 1;
  }
  printf("host sanitizer driver: all checks passed\n");
  return 0;
}
