// combine.cu -- merge of the split-T partials (flash-decoding log-sum-exp merge).
// The partials of (sequence, head) are those of the work items of its head
// group, whose range the split kernel recorded in the workspace's item table.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"),
// closing note: split-T kernels remove the T caps of the CUDA path.  With the
// partials of one (sequence, head) in log2 units, M = max_s m_s and
// w_s = 2^(m_s - M):
//   out = sum_s w_s o_s / sum_s w_s l_s,   lse = ln2 * (M + log2 sum_s w_s l_s).
// One CTA of 256 threads per (head, sequence).  The maxima and weights of the
// splits are computed by all threads together (block reductions), the weights
// kept in shared memory; then thread i of half q sums channels 4i..4i+3 over the
// splits s = q, q+2, ... in order, with eight splits' loads in flight, and the
// two halves are added (half 0 first), so the result is reproducible.
#include "kv8_common.cuh"

namespace kv8 {
namespace {

constexpr int CT = 256;         // threads per CTA
constexpr int WCHUNK = 1024;    // split weights held in shared memory at a time

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  const float r = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])),
                        fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7])));
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(CT) combine_kernel(DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  __shared__ long long s_first, s_count;
  __shared__ float red[8];
  __shared__ float4 half1[128];
  __shared__ float wsh[WCHUNK];
  if (threadIdx.x == 0) {
    const int64_t* e = a.seg + ((int64_t)b * a.plan.n_hg + h / a.plan.hg) * 2;
    s_first = e[0];
    s_count = e[1];
  }
  __syncthreads();
  const int64_t first = s_first, ns = s_count;
  const int hl = h % a.plan.hg, hg = a.plan.hg;
  auto part = [&](int64_t s) -> int64_t { return (first + s) * hg + hl; };

  float M = -INFINITY;
  for (int64_t s = threadIdx.x; s < ns; s += CT) M = fmaxf(M, a.ws_m[part(s)]);
  M = block_max(M, red);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float Lsum = 0.f;  // thread 0's running denominator, in split order
  if (M != -INFINITY) {
    for (int64_t c0 = 0; c0 < ns; c0 += WCHUNK) {
      const int n = (int)((ns - c0) < WCHUNK ? (ns - c0) : WCHUNK);
      for (int s = threadIdx.x; s < n; s += CT) {
        const float ms = a.ws_m[part(c0 + s)];
        wsh[s] = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      }
      __syncthreads();
      if (threadIdx.x == 0)
        for (int s = 0; s < n; ++s) Lsum += wsh[s] * a.ws_l[part(c0 + s)];
      const int q = threadIdx.x >> 7;
      const float4* o = reinterpret_cast<const float4*>(a.ws_o) + (threadIdx.x & 127);
      int s = q;
      for (; s + 14 < n; s += 16) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = o[part(c0 + s + 2 * k) * (DL / 4)];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float w = wsh[s + 2 * k];
          acc.x += w * v[k].x; acc.y += w * v[k].y; acc.z += w * v[k].z; acc.w += w * v[k].w;
        }
      }
      for (; s < n; s += 2) {
        const float w = wsh[s];
        const float4 v = o[part(c0 + s) * (DL / 4)];
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
      }
      __syncthreads();
    }
  }
  if (threadIdx.x >= 128) half1[threadIdx.x - 128] = acc;
  if (threadIdx.x == 0) red[0] = Lsum;
  __syncthreads();
  if (threadIdx.x >= 128) return;
  const float4 a1 = half1[threadIdx.x];
  acc.x += a1.x; acc.y += a1.y; acc.z += a1.z; acc.w += a1.w;
  const float L = red[0];
  const float inv = (L > 0.f) ? 1.0f / L : 0.f;
  float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  reinterpret_cast<float4*>(a.out + ((int64_t)b * a.H + h) * DL)[threadIdx.x] = r;
  if (a.lse != nullptr && threadIdx.x == 0)
    a.lse[(int64_t)b * a.H + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.H, a.B);
  combine_kernel<<<grid, CT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kv8
