// quantize.cu -- kv8_quantize_rows: f32 latent rows -> e4m3 codes + per-segment
// f32 scales.  KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with
// .coli_kv v2"), PR description, c/kv_fp8.h item: per-row quantizer with a
// subnormal-amax guard, RNE encoding saturating at +-448, signed zero kept,
// NaN stored as inert 0; opening paragraph / expanded summary: one f32
// amax/448 scale for Lc and one for Rc.
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
  for (int64_t r = warp_global; r < n_rows; r += n_warps) {
    const int64_t slot = dst_slot ? __ldg(&dst_slot[r]) : r;
    if (slot < 0 || slot >= n_slots) continue;  // warp-uniform
    const float4* row = reinterpret_cast<const float4*>(src + r * stride);
    float4 L[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) L[k] = __ldcs(&row[lane * 4 + k]);
    float4 R = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < 16) R = __ldcs(&row[128 + lane]);

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

}  // namespace

cudaError_t launch_quantize(const float* src, int64_t n_rows, int64_t stride,
                            const int64_t* dst_slot, uint8_t* codes, float* scales,
                            int64_t n_slots, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t want = (n_rows + QWARPS - 1) / QWARPS;
  const int64_t cap = (int64_t)NUM_SMS * 8;  // 8 CTAs of 8 warps per SM: 64 rows in flight
  const int grid = (int)(want < cap ? want : cap);
  quantize_rows_kernel<<<grid, QWARPS * 32, 0, s>>>(src, n_rows, stride, dst_slot, codes, scales,
                                                    n_slots);
  return cudaGetLastError();
}

}  // namespace kv8
