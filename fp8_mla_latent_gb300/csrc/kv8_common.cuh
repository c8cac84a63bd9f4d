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

// Page-table lookup: cache slot of token t of sequence b, or -1 if the block
// table entry is out of range (the error word records it).
__device__ __forceinline__ int64_t slot_of(const DecodeArgs& a, int b, int64_t t) {
  if (a.block_table == nullptr) return t;
  const int32_t blk = __ldg(&a.block_table[(int64_t)b * a.max_blocks + (t >> 6)]);
  if (blk < 0 || (int64_t)blk >= a.n_blocks) {
    atomicOr(a.err, ERR_BLOCK_TABLE);
    return -1;
  }
  return (int64_t)blk * PAGE + (t & (PAGE - 1));
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

}  // namespace kv8
