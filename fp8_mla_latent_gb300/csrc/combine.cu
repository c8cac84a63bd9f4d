// combine.cu -- merge of the split-T partials (flash-decoding log-sum-exp merge).
// The partials of (sequence, head) are those of the work items of its head
// group, found from the sequence lengths exactly as the split kernel cut them.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"),
// closing note: split-T kernels remove the T caps of the CUDA path.  With the
// partials of one (sequence, head) in log2 units, M = max_s m_s and
// w_s = 2^(m_s - M):
//   out = sum_s w_s o_s / sum_s w_s l_s,   lse = ln2 * (M + log2 sum_s w_s l_s).
// One CTA of 128 threads per (head, sequence); thread i owns channels 4i..4i+3.
#include "kv8_common.cuh"

namespace kv8 {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  __shared__ long long s_first, s_count;
  if (threadIdx.x < 32) {
    int64_t f, c;
    item_range(a, b, h / a.plan.hg, f, c);
    if (threadIdx.x == 0) {
      s_first = f;
      s_count = c;
    }
  }
  __syncthreads();
  const int64_t first = s_first, ns = s_count;
  const int hl = h % a.plan.hg;
  float M = -INFINITY;
  for (int64_t s = 0; s < ns; ++s) M = fmaxf(M, a.ws_m[(first + s) * a.plan.hg + hl]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int64_t s = 0; s < ns; ++s) {
      const int64_t part = (first + s) * a.plan.hg + hl;
      const float ms = a.ws_m[part];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      L += w * a.ws_l[part];
      const float4 o = reinterpret_cast<const float4*>(a.ws_o + part * DL)[threadIdx.x];
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
  }
  const float inv = (L > 0.f) ? 1.0f / L : 0.f;
  float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  reinterpret_cast<float4*>(a.out + ((int64_t)b * a.H + h) * DL)[threadIdx.x] = r;
  if (a.lse != nullptr && threadIdx.x == 0)
    a.lse[(int64_t)b * a.H + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.H, a.B);
  combine_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kv8
