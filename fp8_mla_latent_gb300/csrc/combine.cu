// combine.cu -- merge of the split-T partials (flash-decoding log-sum-exp merge).
// The partials of (sequence, head) are those of the work items of its head
// group, whose range the split kernel recorded in the workspace's item table.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"),
// closing note: split-T kernels remove the T caps of the CUDA path.  With the
// partials of one (sequence, head) in log2 units, M = max_s m_s and
// w_s = 2^(m_s - M):
//   out = sum_s w_s o_s / sum_s w_s l_s,   lse = ln2 * (M + log2 sum_s w_s l_s).
// Two forms.  With fewer than 1024 (sequence, head) pairs, one CTA of 256
// threads per pair (described above the kernel).  Otherwise one warp per pair,
// eight per CTA, no block barriers: the warp takes M by a butterfly over its
// lanes' strided maxima, then walks the splits in order, every lane computing the
// same weight w_s and running denominator (so the sum order is fixed and no
// reduction is needed) while it accumulates its 16 channels (four 16-byte pieces,
// 512 B per warp load, coalesced); the splits' loads go out two splits ahead of
// their use.
// Both forms are deterministic.
#include "kv8_common.cuh"

namespace kv8 {
namespace {

constexpr int CT = 256;                 // threads per CTA (warp form: eight pairs)
constexpr int WPC = CT / 32;
constexpr int AHEAD = 2;                // splits whose loads are in flight per warp
// Few (sequence, head) pairs come with many splits each (a long sequence cut into
// one wave of items): a CTA of 256 threads per pair then keeps more loads in
// flight.  Many pairs come with few splits: one warp per pair.
constexpr int64_t WARP_PATH_MIN = 1024;

// CTA form: 256 threads, two groups of 128; thread i of group q holds channels
// 4i..4i+3 of the splits s = q (mod 2).  Each pass takes up to PASS splits: all
// of a thread's partial loads (PASS / 2 of them) and the splits' (m, l) go out
// together, then the block maximum, the weights 2^(m_s - M) and the denominator
// (thread 0, in split order) come from shared memory, each group sums its splits
// in order, and the two groups are added in order.  Two CTAs fit on an SM, so
// 128 heads of two sequences run in one wave.  Deterministic.
constexpr int CT4 = 256;
constexpr int PASS = 40;
constexpr int PER = PASS / 2;   // partial loads per thread per pass

__global__ void __launch_bounds__(CT4) combine_cta_kernel(DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  __shared__ long long s_first, s_count;
  __shared__ float red[16];
  __shared__ float ms[PASS], ls[PASS], wsh[PASS];
  __shared__ float4 grp[128];
  if (threadIdx.x == 0) {
    const int64_t* e = a.seg + ((int64_t)b * a.plan.n_hg + h / a.plan.hg) * 2;
    s_first = e[0];
    s_count = e[1];
  }
  __syncthreads();
  const int64_t first = s_first, ns = s_count;
  const int hl = h % a.plan.hg, hg = a.plan.hg;
  auto part = [&](int64_t s) -> int64_t { return (first + s) * hg + hl; };
  const int q = threadIdx.x >> 7, i = threadIdx.x & 127;  // group, channel quad
  const float4* o = reinterpret_cast<const float4*>(a.ws_o) + i;

  // the maximum over every split first (one pass over m)
  float M = -INFINITY;
  for (int64_t s = threadIdx.x; s < ns; s += CT4) M = fmaxf(M, a.ws_m[part(s)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int k = 1; k < CT4 / 32; ++k) M = fmaxf(M, red[k]);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;  // thread 0's denominator, in split order
  for (int64_t c0 = 0; M != -INFINITY && c0 < ns; c0 += PASS) {
    const int n = (int)((ns - c0) < PASS ? (ns - c0) : PASS);
    float4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int s = q + 2 * k;
      v[k] = s < n ? o[part(c0 + s) * (DL / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();  // the previous pass is done with ms / ls / wsh
    if (threadIdx.x < n) {
      ms[threadIdx.x] = a.ws_m[part(c0 + threadIdx.x)];
      ls[threadIdx.x] = a.ws_l[part(c0 + threadIdx.x)];
    }
    __syncthreads();
    if (threadIdx.x < n) wsh[threadIdx.x] = ms[threadIdx.x] == -INFINITY ? 0.f : exp2f(ms[threadIdx.x] - M);
    __syncthreads();
    if (threadIdx.x == 0)
      for (int s = 0; s < n; ++s) L += wsh[s] * ls[s];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int s = q + 2 * k;
      if (s < n) {
        const float w = wsh[s];
        acc.x += w * v[k].x; acc.y += w * v[k].y; acc.z += w * v[k].z; acc.w += w * v[k].w;
      }
    }
  }
  if (q > 0) grp[i] = acc;
  if (threadIdx.x == 0) red[0] = L;
  __syncthreads();
  if (q > 0) return;
  const float4 x = grp[i];
  acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
  L = red[0];
  const float inv = (L > 0.f) ? 1.0f / L : 0.f;
  reinterpret_cast<float4*>(a.out + ((int64_t)b * a.H + h) * DL)[i] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (a.lse != nullptr && i == 0)
    a.lse[(int64_t)b * a.H + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

__global__ void __launch_bounds__(CT) combine_warp_kernel(DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = (int64_t)blockIdx.x * WPC + warp;
  if (bh >= (int64_t)a.B * a.H) return;
  const int b = (int)(bh / a.H), h = (int)(bh % a.H);
  const int64_t* e = a.seg + ((int64_t)b * a.plan.n_hg + h / a.plan.hg) * 2;
  const int64_t first = e[0], ns = e[1];
  const int hl = h % a.plan.hg, hg = a.plan.hg;
  auto part = [&](int64_t s) -> int64_t { return (first + s) * hg + hl; };
  const float4* o = reinterpret_cast<const float4*>(a.ws_o) + lane;

  float M = -INFINITY;
  for (int64_t s = lane; s < ns; s += 32) M = fmaxf(M, a.ws_m[part(s)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    // v[d][k]: split s + d, piece k; AHEAD splits in flight ahead of their use
    float4 v[AHEAD][4];
    float mv[AHEAD], lv[AHEAD];
    auto fetch = [&](int64_t s, int d) {
      if (s < ns) {
        const int64_t p = part(s);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[d][k] = o[p * (DL / 4) + 32 * k];
        mv[d] = a.ws_m[p];
        lv[d] = a.ws_l[p];
      }
    };
#pragma unroll
    for (int d = 0; d < AHEAD; ++d) fetch(d, d);
    for (int64_t s = 0; s < ns; s += AHEAD) {
#pragma unroll
      for (int d = 0; d < AHEAD; ++d) {
        if (s + d < ns) {
          const float w = (mv[d] == -INFINITY) ? 0.f : exp2f(mv[d] - M);
          L += w * lv[d];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[k].x += w * v[d][k].x; acc[k].y += w * v[d][k].y;
            acc[k].z += w * v[d][k].z; acc[k].w += w * v[d][k].w;
          }
          fetch(s + d + AHEAD, d);
        }
      }
    }
  }
  const float inv = (L > 0.f) ? 1.0f / L : 0.f;
  float4* out = reinterpret_cast<float4*>(a.out + ((int64_t)b * a.H + h) * DL) + lane;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out[32 * k] = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
  if (a.lse != nullptr && lane == 0)
    a.lse[(int64_t)b * a.H + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  const int64_t warps = (int64_t)a.B * a.H;
  if (warps >= WARP_PATH_MIN) {
    combine_warp_kernel<<<(unsigned)((warps + WPC - 1) / WPC), CT, 0, s>>>(a);
  } else {
    dim3 grid(a.H, a.B);
    combine_cta_kernel<<<grid, CT4, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kv8
