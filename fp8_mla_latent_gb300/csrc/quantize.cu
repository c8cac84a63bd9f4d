// quantize.cu -- kv8_quantize_rows: f32 latent rows -> e4m3 codes + per-segment
// f32 scales.  KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description, c/kv_fp8.h item: per-row quantizer with a
// subnormal-amax guard, RNE encoding saturating at +-448, signed zero kept,
// NaN stored as inert 0; opening paragraph / expanded summary: one f32
// amax/448 scale for Lc and one for Rc.
//
// produce_rows_kernel is the fused producer in front of it (PR description,
// attention_rows item: the producer quantizes the new row once normalised and
// rotated): RMS norm of Lc with a weight, rotation of the Rc pairs (2j, 2j+1) by the angle of
// the row's position (cosine and sine tabulated by the caller), then the same
// quantization.  Its f32 operations are rounded once each, in a fixed order (the
// sum of squares: lane partial sums in index order, then an xor butterfly), so
// the codes are reproducible bit for bit.
//
// One warp per row.  Lane l reads Lc floats [16l, 16l+16) as four 16-byte loads
// and, for l < 16, Rc floats [512+4l, 512+4l+4) as one; it writes its 16 Lc codes
// as one 16-byte store and its 4 Rc codes as one 4-byte store.  A row moves
// 2304 B in and 584 B out: the kernel is a pure HBM stream.
#include "kv8_common.cuh"

namespace kv8 {
namespace {

constexpr int QWARPS = 8;  // rows in flight per CTA

__device__ __forceinline__ float absmax_nonnan(float acc, float x) {
  // fmaxf returns the non-NaN operand, so NaN never raises the maximum
  return fmaxf(acc, fabsf(x));
}

__device__ __forceinline__ uint8_t zero_code(float x) {
  // guard path: signed zero, NaN -> 0x00
  return (!isnan(x) && signbit(x)) ? 0x80u : 0x00u;
}

// Encode 4 floats given the segment's inverse scale (or the guard).
__device__ __forceinline__ uint32_t encode4(float4 v, float inv, bool guard) {
  if (guard) {
    return (uint32_t)zero_code(v.x) | ((uint32_t)zero_code(v.y) << 8) |
           ((uint32_t)zero_code(v.z) << 16) | ((uint32_t)zero_code(v.w) << 24);
  }
  // product rounded once (no contraction: __fmul_rn), NaN replaced by +0
  float p0 = __fmul_rn(v.x, inv), p1 = __fmul_rn(v.y, inv);
  float p2 = __fmul_rn(v.z, inv), p3 = __fmul_rn(v.w, inv);
  p0 = isnan(p0) ? 0.0f : p0;
  p1 = isnan(p1) ? 0.0f : p1;
  p2 = isnan(p2) ? 0.0f : p2;
  p3 = isnan(p3) ? 0.0f : p3;
  return (uint32_t)f32x2_to_e4m3x2(p0, p1) | ((uint32_t)f32x2_to_e4m3x2(p2, p3) << 16);
}

__global__ void __launch_bounds__(QWARPS * 32)
quantize_rows_kernel(const float* __restrict__ src, int64_t n_rows, int64_t stride,
                     const int64_t* __restrict__ dst_slot, uint8_t* __restrict__ codes,
                     float* __restrict__ scales, int64_t n_slots) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t)blockIdx.x * QWARPS + (threadIdx.x >> 5);
  const int64_t n_warps = (int64_t)gridDim.x * QWARPS;
  // the row's data is requested together with its slot (one round trip per row)
  for (int64_t r = warp_global; r < n_rows; r += n_warps) {
    const int64_t slot = dst_slot ? __ldg(&dst_slot[r]) : r;
    const float4* row = reinterpret_cast<const float4*>(src + r * stride);
    float4 L[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) L[k] = __ldcs(&row[lane * 4 + k]);
    float4 R = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < 16) R = __ldcs(&row[128 + lane]);
    if (slot < 0 || slot >= n_slots) continue;  // warp-uniform

    float aL = 0.0f, aR = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      aL = absmax_nonnan(aL, L[k].x); aL = absmax_nonnan(aL, L[k].y);
      aL = absmax_nonnan(aL, L[k].z); aL = absmax_nonnan(aL, L[k].w);
    }
    aR = absmax_nonnan(aR, R.x); aR = absmax_nonnan(aR, R.y);
    aR = absmax_nonnan(aR, R.z); aR = absmax_nonnan(aR, R.w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      aL = fmaxf(aL, __shfl_xor_sync(0xffffffffu, aL, o));
      aR = fmaxf(aR, __shfl_xor_sync(0xffffffffu, aR, o));
    }
    const float sL = __fdiv_rn(aL, 448.0f), sR = __fdiv_rn(aR, 448.0f);
    const float iL = __fdiv_rn(448.0f, aL), iR = __fdiv_rn(448.0f, aR);
    const bool gL = !isfinite(iL), gR = !isfinite(iR);

    uint4 cl;
    cl.x = encode4(L[0], iL, gL);
    cl.y = encode4(L[1], iL, gL);
    cl.z = encode4(L[2], iL, gL);
    cl.w = encode4(L[3], iL, gL);
    uint8_t* dst = codes + slot * D;
    *reinterpret_cast<uint4*>(dst + lane * 16) = cl;
    if (lane < 16) *reinterpret_cast<uint32_t*>(dst + DL + lane * 4) = encode4(R, iR, gR);
    if (lane == 0) *reinterpret_cast<float2*>(scales + slot * 2) = make_float2(sL, sR);
  }
}

// Encode the two Rc values of one rotary pair (the producer's lane layout).
__device__ __forceinline__ uint32_t encode2(float a, float b, float inv, bool guard) {
  if (guard) return (uint32_t)zero_code(a) | ((uint32_t)zero_code(b) << 8);
  float p0 = __fmul_rn(a, inv), p1 = __fmul_rn(b, inv);
  p0 = isnan(p0) ? 0.0f : p0;
  p1 = isnan(p1) ? 0.0f : p1;
  return (uint32_t)f32x2_to_e4m3x2(p0, p1);
}

__global__ void __launch_bounds__(QWARPS * 32)
produce_rows_kernel(const float* __restrict__ src, int64_t n_rows, int64_t stride,
                    const float* __restrict__ weight, float eps,
                    const int64_t* __restrict__ positions, const float* __restrict__ rope_cos,
                    const float* __restrict__ rope_sin, int64_t max_pos,
                    const int64_t* __restrict__ dst_slot, uint8_t* __restrict__ codes,
                    float* __restrict__ scales, int64_t n_slots, unsigned* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t)blockIdx.x * QWARPS + (threadIdx.x >> 5);
  const int64_t n_warps = (int64_t)gridDim.x * QWARPS;
  // the lane's 16 norm weights
  float4 W[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) W[k] = __ldg(reinterpret_cast<const float4*>(weight) + lane * 4 + k);
  // Software pipeline: the slot and position of the next row are loaded while
  // this row is processed, and a row's data is requested together with its
  // rotation table entries, so each row costs one round trip to memory.
  int64_t r = warp_global;
  int64_t slot = 0, pos = 0;
  if (r < n_rows) {
    slot = dst_slot ? __ldg(&dst_slot[r]) : r;
    pos = __ldg(&positions[r]);
  }
  for (; r < n_rows; r += n_warps) {
    const bool valid = !(slot < 0 || slot >= n_slots || pos < 0 || pos >= max_pos);  // warp-uniform
    const int64_t pc = valid ? pos : 0;
    const float4* row = reinterpret_cast<const float4*>(src + r * stride);
    float4 L[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) L[k] = __ldcs(&row[lane * 4 + k]);
    const float2 X = __ldcs(reinterpret_cast<const float2*>(src + r * stride + DL) + lane);
    const float c = __ldg(&rope_cos[pc * (DR / 2) + lane]), sn = __ldg(&rope_sin[pc * (DR / 2) + lane]);
    const int64_t rn = r + n_warps;
    int64_t slot_n = 0, pos_n = 0;
    if (rn < n_rows) {
      slot_n = dst_slot ? __ldg(&dst_slot[rn]) : rn;
      pos_n = __ldg(&positions[rn]);
    }
    const int64_t slot_c = slot;
    slot = slot_n;
    if (!valid) {
      if (lane == 0 && err != nullptr && (pos < 0 || pos >= max_pos)) atomicOr(err, 1u);
      pos = pos_n;
      continue;
    }
    pos = pos_n;

    // RMS norm: sum of squares in the fixed order, then y = (x * inv) * w
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ss = __fadd_rn(ss, __fmul_rn(L[k].x, L[k].x));
      ss = __fadd_rn(ss, __fmul_rn(L[k].y, L[k].y));
      ss = __fadd_rn(ss, __fmul_rn(L[k].z, L[k].z));
      ss = __fadd_rn(ss, __fmul_rn(L[k].w, L[k].w));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float inv_rms =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / 512.0f), eps)));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      L[k].x = __fmul_rn(__fmul_rn(L[k].x, inv_rms), W[k].x);
      L[k].y = __fmul_rn(__fmul_rn(L[k].y, inv_rms), W[k].y);
      L[k].z = __fmul_rn(__fmul_rn(L[k].z, inv_rms), W[k].z);
      L[k].w = __fmul_rn(__fmul_rn(L[k].w, inv_rms), W[k].w);
    }
    // rotary pair of this lane
    const float y0 = __fsub_rn(__fmul_rn(X.x, c), __fmul_rn(X.y, sn));
    const float y1 = __fadd_rn(__fmul_rn(X.x, sn), __fmul_rn(X.y, c));

    // quantize (as quantize_rows_kernel)
    float aL = 0.0f, aR = absmax_nonnan(absmax_nonnan(0.0f, y0), y1);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      aL = absmax_nonnan(aL, L[k].x); aL = absmax_nonnan(aL, L[k].y);
      aL = absmax_nonnan(aL, L[k].z); aL = absmax_nonnan(aL, L[k].w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      aL = fmaxf(aL, __shfl_xor_sync(0xffffffffu, aL, o));
      aR = fmaxf(aR, __shfl_xor_sync(0xffffffffu, aR, o));
    }
    const float sL = __fdiv_rn(aL, 448.0f), sR = __fdiv_rn(aR, 448.0f);
    const float iL = __fdiv_rn(448.0f, aL), iR = __fdiv_rn(448.0f, aR);
    const bool gL = !isfinite(iL), gR = !isfinite(iR);
    uint4 cl;
    cl.x = encode4(L[0], iL, gL);
    cl.y = encode4(L[1], iL, gL);
    cl.z = encode4(L[2], iL, gL);
    cl.w = encode4(L[3], iL, gL);
    uint8_t* dst = codes + slot_c * D;
    *reinterpret_cast<uint4*>(dst + lane * 16) = cl;
    *reinterpret_cast<uint16_t*>(dst + DL + lane * 2) = (uint16_t)encode2(y0, y1, iR, gR);
    if (lane == 0) *reinterpret_cast<float2*>(scales + slot_c * 2) = make_float2(sL, sR);
  }
}

}  // namespace

cudaError_t launch_quantize(const float* src, int64_t n_rows, int64_t stride,
                            const int64_t* dst_slot, uint8_t* codes, float* scales,
                            int64_t n_slots, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t want = (n_rows + QWARPS - 1) / QWARPS;
  // as many CTAs as are resident at once (the loop strides over the rest)
  static std::atomic<int> memo[MAX_DEVICES];
  int per_sm = 0;
  const cudaError_t e = per_device(memo, [](int* v) {
    int n = 0;
    const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_rows_kernel, QWARPS * 32, 0);
    *v = n < 1 ? 1 : n;
    return r;
  }, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t cap = (int64_t)NUM_SMS * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  quantize_rows_kernel<<<grid, QWARPS * 32, 0, s>>>(src, n_rows, stride, dst_slot, codes, scales,
                                                    n_slots);
  return cudaGetLastError();
}

}  // namespace kv8

namespace kv8 {

cudaError_t launch_produce(const float* src, int64_t n_rows, int64_t stride, const float* weight,
                          float eps, const int64_t* positions, const float* rope_cos,
                          const float* rope_sin, int64_t max_pos, const int64_t* dst_slot,
                          uint8_t* codes, float* scales, int64_t n_slots, unsigned* err,
                          cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t want = (n_rows + QWARPS - 1) / QWARPS;
  // as many CTAs as are resident at once (the loop strides over the rest)
  static std::atomic<int> memo[MAX_DEVICES];
  int per_sm = 0;
  const cudaError_t e = per_device(memo, [](int* v) {
    int n = 0;
    const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, produce_rows_kernel, QWARPS * 32, 0);
    *v = n < 1 ? 1 : n;
    return r;
  }, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t cap = (int64_t)NUM_SMS * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  produce_rows_kernel<<<grid, QWARPS * 32, 0, s>>>(src, n_rows, stride, weight, eps, positions,
                                                   rope_cos, rope_sin, max_pos, dst_slot, codes,
                                                   scales, n_slots, err);
  return cudaGetLastError();
}

}  // namespace kv8
