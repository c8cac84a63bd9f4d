// wuv.cu -- the W_UV epilogue of absorbed MLA decode: the per-head projection of
// the latent context to the value head, y[b][h][v] = sum_d o[b][h][d] W_UV[h][d][v].
//
// KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
// description: in the absorbed attention the latent is key and value at once, so
// the attention's context is a latent vector per head and the value projection
// follows it.
//
// Decode has one query row per sequence, so the work is B x H dot products of
// length 512 per output column: the weight stream (H x 512 x V bf16, 16 MB at
// H = V = 128) bounds it, not arithmetic.  One CTA per (head, 128 output
// columns), the sequences' context rows in shared memory.  When V is a multiple
// of 8 (and the weights 16-byte aligned), thread (r, g) of 512 owns columns
// 8g..8g+7 and the latent rows d = r, r+32, ...: one 16-byte load brings 8
// weights, all sixteen rows' loads in flight; the 32 row groups are then added in a
// fixed order through shared memory.  Otherwise thread (k, v) sums half k of the
// latent rows for column v with 2-byte loads.  The bf16 -> f32 conversion is
// exact.
#include "kv8_common.cuh"

namespace kv8 {
namespace {

constexpr int WT = 256;       // threads: 2 halves of the latent rows x 128 columns
constexpr int BMAX = 16;      // sequences per pass (accumulators per thread)

__global__ void __launch_bounds__(WT) wuv_kernel(const float* __restrict__ o,
                                                 const uint16_t* __restrict__ w, int B, int H,
                                                 int V, float* __restrict__ y) {
  const int h = blockIdx.x;
  const int v = blockIdx.y * 128 + (threadIdx.x & 127);
  const int half = threadIdx.x >> 7;
  __shared__ float osh[BMAX][DL];
  __shared__ float part[BMAX][128];
  const uint16_t* wh = w + (int64_t)h * DL * V;
  for (int b0 = 0; b0 < B; b0 += BMAX) {
    const int nb = (B - b0) < BMAX ? (B - b0) : BMAX;
    for (int i = threadIdx.x; i < nb * DL; i += WT) {
      const int bb = i / DL, d = i % DL;
      osh[bb][d] = o[((int64_t)(b0 + bb) * H + h) * DL + d];
    }
    __syncthreads();
    float acc[BMAX];
#pragma unroll
    for (int k = 0; k < BMAX; ++k) acc[k] = 0.f;
    if (v < V) {
      const int d0 = half * (DL / 2);
#pragma unroll 4
      for (int d = d0; d < d0 + DL / 2; ++d) {
        const float wf = __uint_as_float((uint32_t)__ldg(&wh[(int64_t)d * V + v]) << 16);
#pragma unroll
        for (int k = 0; k < BMAX; ++k)
          if (k < nb) acc[k] = fmaf(osh[k][d], wf, acc[k]);
      }
    }
    if (half == 1) {
#pragma unroll
      for (int k = 0; k < BMAX; ++k) part[k][threadIdx.x & 127] = acc[k];
    }
    __syncthreads();
    if (half == 0 && v < V) {
#pragma unroll
      for (int k = 0; k < BMAX; ++k)
        if (k < nb) y[((int64_t)(b0 + k) * H + h) * V + v] = acc[k] + part[k][threadIdx.x];
    }
    __syncthreads();
  }
}

constexpr int VB = 4;     // sequences per pass of the vector path
constexpr int VT = 512;   // threads of the vector path: 32 latent row groups x 16 column groups
constexpr int VR = VT / 16;
constexpr int V8_SMEM = (VB * DL + VR * VB * 128) * 4;  // context rows + partial sums

__global__ void __launch_bounds__(VT) wuv8_kernel(const float* __restrict__ o,
                                                  const uint16_t* __restrict__ w, int B, int H,
                                                  int V, float* __restrict__ y) {
  const int h = blockIdx.x;
  const int g = threadIdx.x & 15, r = threadIdx.x >> 4;  // column group, latent row group
  const int v0 = blockIdx.y * 128 + g * 8;
  extern __shared__ float wsm[];
  float (*osh)[DL] = reinterpret_cast<float (*)[DL]>(wsm);
  float (*part)[VB][128] = reinterpret_cast<float (*)[VB][128]>(wsm + VB * DL);
  const uint16_t* wh = w + (int64_t)h * DL * V;
  for (int b0 = 0; b0 < B; b0 += VB) {
    const int nb = (B - b0) < VB ? (B - b0) : VB;
    for (int i = threadIdx.x; i < nb * DL; i += VT) {
      const int bb = i / DL, d = i % DL;
      osh[bb][d] = o[((int64_t)(b0 + bb) * H + h) * DL + d];
    }
    __syncthreads();
    float acc[VB][8];
#pragma unroll
    for (int k = 0; k < VB; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[k][j] = 0.f;
    if (v0 < V) {
      // all DL / VR = 16 of this thread's weight rows in flight at once
      uint4 q[DL / VR];
#pragma unroll
      for (int i = 0; i < DL / VR; ++i)
        q[i] = __ldg(reinterpret_cast<const uint4*>(wh + (int64_t)(r + i * VR) * V + v0));
#pragma unroll
      for (int i = 0; i < DL / VR; ++i) {
        const int d = r + i * VR;
        const uint32_t u[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
        float wf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wf[2 * j] = __uint_as_float(u[j] << 16);
          wf[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
        }
#pragma unroll
        for (int k = 0; k < VB; ++k) {
          if (k < nb) {
            const float ob = osh[k][d];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[k][j] = fmaf(ob, wf[j], acc[k][j]);
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < VB; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[r][k][g * 8 + j] = acc[k][j];
    __syncthreads();
    // thread t < nb * 128: column t % 128 of sequence t / 128, row groups in order
    for (int t = threadIdx.x; t < nb * 128; t += VT) {
      const int k = t >> 7, c = t & 127;
      const int v = blockIdx.y * 128 + c;
      float sum = part[0][k][c];
#pragma unroll
      for (int rr = 1; rr < VR; ++rr) sum += part[rr][k][c];
      if (v < V) y[((int64_t)(b0 + k) * H + h) * V + v] = sum;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_wuv(const float* o, const uint16_t* w, int B, int H, int V, float* y,
                       cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  dim3 grid(H, (V + 127) / 128);
  if (V % 8 == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
    static std::atomic<int> memo[MAX_DEVICES];
    int done = 0;
    const cudaError_t e = per_device(memo, [](int* v) {
      *v = 1;
      return cudaFuncSetAttribute(wuv8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, V8_SMEM);
    }, &done);
    if (e != cudaSuccess) return e;
    wuv8_kernel<<<grid, VT, V8_SMEM, s>>>(o, w, B, H, V, y);
  }
  else
    wuv_kernel<<<grid, WT, 0, s>>>(o, w, B, H, V, y);
  return cudaGetLastError();
}

}  // namespace kv8
