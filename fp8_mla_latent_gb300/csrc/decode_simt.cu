// decode_simt.cu -- CUDA-core split-T absorbed MLA decode over the e4m3 cache.
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"),
// PR description: the latent is key and value at once; the score and context
// loops decode as they go, each row scale applied outside its dot product; closing
// note: split-T kernels for long caches.
//
// One CTA per work item (sequence, head group of HG_SIMT heads, token range);
// 8 warps per CTA.
// Lane l owns latent channels [16l, 16l+16) and RoPE channels [512+2l, 512+2l+2),
// so one token row (576 B) is read by the warp as 32 x 16 B + 32 x 2 B.  Each warp
// walks tokens t0 + w, t0 + w + 8, ... keeping an online softmax per head in log2
// units; the 8 warps are merged in a fixed order through shared memory and the split's partial
// (m, l, o) goes to the workspace for the combine kernel.
//
// This is the kernel for small head counts (and a cross-check of the tensor-core
// kernel): at H >= 16 its FP32 lanes, not HBM, bound it.
#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

constexpr int HG_SIMT = 4;
constexpr int SWARPS = 8;
// Items are cut in units of 32 tokens (one group of four tokens per warp), not
// whole tiles, so that a short cache spreads over many SMs.
constexpr int LOG2_UNIT = 5;
constexpr float LOG2E = 1.4426950408889634f;

__global__ void __launch_bounds__(SWARPS * 32, 1)
decode_simt_kernel(DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ WorkItem s_it;
  __shared__ int s_ok;
  __shared__ int32_t pt[PT_PAGES];  // the item's block-table entries
  if (warp == 0) {
    WorkItem it;
    const bool ok = find_item(a, blockIdx.x, it, LOG2_UNIT);
    if (lane == 0 && ok) record_segment(a, blockIdx.x, it);
    if (ok) load_page_table(a, it.b, it.t0, it.t1, pt, lane);
    if (lane == 0) {
      s_it = it;
      s_ok = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;  // past the last work item of this call
  const int b = s_it.b, g = s_it.g;
  const int64_t t0 = s_it.t0, t1 = s_it.t1;
  const int h0 = g * HG_SIMT;

  // query slices, pre-multiplied by sm_scale * log2(e) so scores come out in log2 units
  const float c = a.sm_scale * LOG2E;
  float qL[HG_SIMT][16], qR[HG_SIMT][2];
#pragma unroll
  for (int j = 0; j < HG_SIMT; ++j) {
    const int h = h0 + j;
    if (h < a.H) {
      const float4* ql = reinterpret_cast<const float4*>(a.q_lat + ((int64_t)b * a.H + h) * DL);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = __ldg(&ql[lane * 4 + k]);
        qL[j][4 * k] = v.x * c; qL[j][4 * k + 1] = v.y * c;
        qL[j][4 * k + 2] = v.z * c; qL[j][4 * k + 3] = v.w * c;
      }
      const float2 r = __ldg(reinterpret_cast<const float2*>(
          a.q_rope + ((int64_t)b * a.H + h) * DR + 2 * lane));
      qR[j][0] = r.x * c; qR[j][1] = r.y * c;
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) qL[j][k] = 0.f;
      qR[j][0] = qR[j][1] = 0.f;
    }
  }

  float m[HG_SIMT], l[HG_SIMT], o[HG_SIMT][16];
#pragma unroll
  for (int j = 0; j < HG_SIMT; ++j) {
    m[j] = -INFINITY; l[j] = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) o[j][k] = 0.f;
  }

  // Tokens t0 + warp, + 8, + 16, ... in that order, four at a time: the four rows'
  // loads are in flight together (one row at a time is a chain of dependent loads).
  constexpr int AHEAD = 4;
  for (int64_t tb = t0 + warp; tb < t1; tb += AHEAD * SWARPS) {
    uint4 cl[AHEAD];
    uint16_t cr[AHEAD];
    float2 sc[AHEAD];
    bool have[AHEAD];
#pragma unroll
    for (int u = 0; u < AHEAD; ++u) {
      const int64_t t = tb + u * SWARPS;
      const int64_t slot = t < t1 ? item_slot(a, b, t, t0, pt) : -1;  // a bad page reads as empty
      have[u] = slot >= 0;
      if (have[u]) {
        const uint8_t* row = a.codes + slot * D;
        cl[u] = __ldg(reinterpret_cast<const uint4*>(row) + lane);
        cr[u] = __ldg(reinterpret_cast<const uint16_t*>(row + DL) + lane);
        sc[u] = __ldg(reinterpret_cast<const float2*>(a.scales + slot * 2));
      } else {
        cl[u] = make_uint4(0u, 0u, 0u, 0u);
        cr[u] = 0;
        sc[u] = make_float2(0.f, 0.f);
      }
    }
    // the lane partials of all the group's scores, then their sums over the warp
    // together (the butterflies of the sixteen (token, head) pairs interleave)
    float z[AHEAD][HG_SIMT];
#pragma unroll
    for (int u = 0; u < AHEAD; ++u) {
      float v[16], vr[2];
      e4m3x4_to_f32(cl[u].x, v); e4m3x4_to_f32(cl[u].y, v + 4);
      e4m3x4_to_f32(cl[u].z, v + 8); e4m3x4_to_f32(cl[u].w, v + 12);
      {
        const uint32_t h2 = e4m3x2_to_f16x2(cr[u]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        vr[0] = f.x; vr[1] = f.y;
      }
#pragma unroll
      for (int j = 0; j < HG_SIMT; ++j) {
        float dl = 0.f, dr = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) dl = fmaf(qL[j][k], v[k], dl);
        dr = fmaf(qR[j][0], vr[0], dr);
        dr = fmaf(qR[j][1], vr[1], dr);
        z[u][j] = sc[u].x * dl + sc[u].y * dr;  // the row scales, outside the dot products
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < AHEAD; ++u)
#pragma unroll
        for (int j = 0; j < HG_SIMT; ++j) z[u][j] += __shfl_xor_sync(0xffffffffu, z[u][j], off);
    // the online softmax, token by token (in the same order as before)
#pragma unroll
    for (int u = 0; u < AHEAD; ++u) {
      if (!have[u]) continue;
      float v[16];
      e4m3x4_to_f32(cl[u].x, v); e4m3x4_to_f32(cl[u].y, v + 4);
      e4m3x4_to_f32(cl[u].z, v + 8); e4m3x4_to_f32(cl[u].w, v + 12);
#pragma unroll
      for (int j = 0; j < HG_SIMT; ++j) {
        // a new max rescales the running sums (the same in every lane: z is the
        // warp's sum); 2^(m - mn) is 0 on the first token (m = -inf)
        if (z[u][j] > m[j]) {
          const float alpha = ptx::ex2_approx(m[j] - z[u][j]);
          l[j] *= alpha;
#pragma unroll
          for (int k = 0; k < 16; ++k) o[j][k] *= alpha;
          m[j] = z[u][j];
        }
        const float p = ptx::ex2_approx(z[u][j] - m[j]);
        l[j] += p;
        const float w = p * sc[u].x;
#pragma unroll
        for (int k = 0; k < 16; ++k) o[j][k] = fmaf(w, v[k], o[j][k]);
      }
    }
  }

  // merge the 8 warps: the common max, then the rescaled partials of warps w and
  // w + 4 added into buffer w, then the four buffers added in order.  Channel
  // 16 l + k of a head sits at k * 32 + l (the lanes of a warp on distinct banks).
  __shared__ float sm_m[SWARPS][HG_SIMT], sm_l[SWARPS][HG_SIMT];
  __shared__ float sm_o[SWARPS / 2][HG_SIMT][DL];
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < HG_SIMT; ++j) sm_m[warp][j] = m[j];
  }
  __syncthreads();
  float M[HG_SIMT], f[HG_SIMT];
#pragma unroll
  for (int j = 0; j < HG_SIMT; ++j) {
    M[j] = sm_m[0][j];
#pragma unroll
    for (int w = 1; w < SWARPS; ++w) M[j] = fmaxf(M[j], sm_m[w][j]);
    f[j] = (m[j] == -INFINITY) ? 0.f : exp2f(m[j] - M[j]);
    if (lane == 0) sm_l[warp][j] = l[j] * f[j];
  }
  float* buf = &sm_o[warp % (SWARPS / 2)][0][0];
  if (warp < SWARPS / 2) {
#pragma unroll
    for (int j = 0; j < HG_SIMT; ++j)
#pragma unroll
      for (int k = 0; k < 16; ++k) buf[j * DL + k * 32 + lane] = o[j][k] * f[j];
  }
  __syncthreads();
  if (warp >= SWARPS / 2) {
#pragma unroll
    for (int j = 0; j < HG_SIMT; ++j)
#pragma unroll
      for (int k = 0; k < 16; ++k) buf[j * DL + k * 32 + lane] += o[j][k] * f[j];
  }
  __syncthreads();
  // fixed-order sums (no atomics), so results are bitwise reproducible
  const int64_t base = (int64_t)blockIdx.x * HG_SIMT;  // this item's partials
  for (int i = threadIdx.x; i < HG_SIMT * DL; i += blockDim.x) {
    const int j = i / DL, r = i % DL;  // r = k * 32 + l: channel d = 16 l + k
    const float* o0 = &sm_o[0][0][0];
    const float v = (o0[i] + o0[HG_SIMT * DL + i]) + (o0[2 * HG_SIMT * DL + i] + o0[3 * HG_SIMT * DL + i]);
    if (h0 + j < a.H) a.ws_o[(base + j) * DL + (r & 31) * 16 + (r >> 5)] = v;
  }
  if (threadIdx.x < HG_SIMT && h0 + threadIdx.x < a.H) {
    const int j = threadIdx.x;
    float L = 0.f;
    for (int w = 0; w < SWARPS; ++w) L += sm_l[w][j];
    a.ws_m[base + j] = M[j];
    a.ws_l[base + j] = L;
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t s) {
  decode_simt_kernel<<<a.plan.max_items, SWARPS * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kv8
