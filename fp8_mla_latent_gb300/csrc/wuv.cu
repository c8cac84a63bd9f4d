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
// H = V = 128) bounds it, not arithmetic.  When V is a multiple of 8 (and the
// weights 16-byte aligned) the bulk path below streams the weights into shared
// memory on clusters of four CTAs per (head, 128 output columns).  Otherwise one
// CTA per (head, 128 output columns), the sequences' context rows in shared
// memory, and thread (k, v) sums half k of the latent rows for column v with
// 2-byte loads.  The bf16 -> f32 conversion is exact.
#include "kv8_common.cuh"
#include "tc_ptx.cuh"

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

// The bulk path (V a multiple of 8, weights 16-byte aligned).  A cluster of
// SPLIT CTAs takes one (head, block of 128 output columns); CTA q of the cluster
// holds latent rows [128 q, 128 q + 128).  Its weights (at most 32 KB) come in by
// bulk copies into shared memory, in four chunks of 32 rows with a barrier each,
// all in flight at once: a plain-load stream from a few SMs cannot keep enough
// bytes in flight to fill HBM.  Thread (r, g) of 256 owns columns 8g..8g+7 and
// rows 8r..8r+7 of the CTA's quarter; the partial sums are added in a fixed order:
// the two row groups of a warp (a shuffle), then the warps in order, then the
// cluster's CTAs in rank order (read from their shared memory).
constexpr int SPLIT = 4;                // CTAs of a cluster, latent rows each: DL / SPLIT
constexpr int QR = DL / SPLIT;          // 128 latent rows per CTA
constexpr int BT = 256;                 // threads: 16 row groups x 16 column groups
constexpr int BCH = 2;                  // sequences per pass
constexpr int NCHUNK = 4;               // weight chunks (barriers) of QR / NCHUNK rows
constexpr uint64_t WUV_WAIT_NS = 2000000000ull;
constexpr int OFF_W = 0;                                  // [QR][pitch] bf16, pitch <= 256 B
constexpr int OFF_O = OFF_W + QR * 256;                   // [BCH][QR] f32 contexts
constexpr int OFF_PART = OFF_O + BCH * QR * 4;            // [BT / 32][BCH][128] f32
constexpr int OFF_Y = OFF_PART + (BT / 32) * BCH * 128 * 4;  // [BCH][128] f32, this CTA's sums
constexpr int OFF_BAR = OFF_Y + BCH * 128 * 4;
constexpr int BULK_SMEM = OFF_BAR + NCHUNK * 8 + 8;
static_assert(OFF_BAR % 8 == 0 && OFF_O % 16 == 0, "shared-memory layout");

__global__ void __cluster_dims__(SPLIT, 1, 1) __launch_bounds__(BT, 4)
    wuv_bulk_kernel(const float* __restrict__ o, const uint16_t* __restrict__ w, int B, int H,
                    int V, float* __restrict__ y) {
  extern __shared__ __align__(128) uint8_t wsm[];
  const int h = blockIdx.x / SPLIT;
  const uint32_t q = ptx::cluster_rank();
  const int v0 = blockIdx.y * 128;
  const int ncol = (V - v0) < 128 ? (V - v0) : 128;  // a multiple of 8
  const uint32_t pitch = (uint32_t)ncol * 2u;          // bytes per weight row in shared memory
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane & 15, r = (warp << 1) | (lane >> 4);  // column group, row group
  uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + OFF_BAR);
  volatile int* bad = reinterpret_cast<volatile int*>(wsm + OFF_BAR + NCHUNK * 8);
  float* osh = reinterpret_cast<float*>(wsm + OFF_O);
  float* part = reinterpret_cast<float*>(wsm + OFF_PART);
  float* ycta = reinterpret_cast<float*>(wsm + OFF_Y);
  const uint32_t wbase = ptx::smem_u32(wsm + OFF_W);
  const uint16_t* wq = w + ((int64_t)h * DL + q * QR) * V + v0;

  if (threadIdx.x == 0) {
    for (int c = 0; c < NCHUNK; ++c) ptx::mbar_init(&bars[c], 1);
    bad[0] = 0;
    bad[1] = 0;  // never set: the abort flag of the final wait
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0) {
    // chunk c = rows [32 c, 32 c + 32): one copy when the rows are contiguous in
    // global memory (ncol == V), else one per row, lane l taking row 32 c + l
    constexpr int CR = QR / NCHUNK;
    if (lane == 0)
      for (int c = 0; c < NCHUNK; ++c) ptx::mbar_arrive_expect_tx(&bars[c], CR * pitch);
    __syncwarp();
    for (int c = 0; c < NCHUNK; ++c) {
      if (ncol == V) {
        if (lane == 0)
          ptx::bulk_load_g2s(wbase + c * CR * pitch, wq + (int64_t)c * CR * V, CR * pitch, &bars[c]);
      } else {
        const int row = c * CR + lane;
        ptx::bulk_load_g2s(wbase + row * pitch, wq + (int64_t)row * V, pitch, &bars[c]);
      }
    }
  }
  // this warp's rows 8r..8r+7 lie in chunk r / 4 (= warp / 2)
  const int chunk = warp >> 1;
  bool ready = false;
  const bool active = g * 8 < ncol;
  for (int b0 = 0; b0 < B; b0 += BCH) {
    const int nb = (B - b0) < BCH ? (B - b0) : BCH;
    for (int i = threadIdx.x; i < BCH * QR; i += BT) {
      const int k = i / QR, d = i % QR;
      osh[i] = k < nb ? __ldg(o + ((int64_t)(b0 + k) * H + h) * DL + q * QR + d) : 0.f;
    }
    __syncthreads();
    if (!ready) {
      ready = true;
      if (!ptx::mbar_wait(&bars[chunk], 0, bad, WUV_WAIT_NS)) *bad = 1;
    }
    float acc[BCH][8];
#pragma unroll
    for (int k = 0; k < BCH; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[k][j] = 0.f;
    if (active) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = r * 8 + i;
        const uint4 u4 = lds128(wbase + d * pitch + g * 16);
        const uint32_t u[4] = {u4.x, u4.y, u4.z, u4.w};
        float wf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wf[2 * j] = __uint_as_float(u[j] << 16);
          wf[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
        }
#pragma unroll
        for (int k = 0; k < BCH; ++k) {
          const float ob = osh[k * QR + d];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[k][j] = fmaf(ob, wf[j], acc[k][j]);
        }
      }
    }
    // row groups 2w and 2w + 1, then the warps in order
#pragma unroll
    for (int k = 0; k < BCH; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[k][j] += __shfl_xor_sync(0xffffffffu, acc[k][j], 16);
    if (lane < 16) {
#pragma unroll
      for (int k = 0; k < BCH; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) part[(warp * BCH + k) * 128 + g * 8 + j] = acc[k][j];
    }
    __syncthreads();
    for (int t = threadIdx.x; t < BCH * 128; t += BT) {
      float sum = part[t];
#pragma unroll
      for (int ww = 1; ww < BT / 32; ++ww) sum += part[ww * BCH * 128 + t];
      ycta[t] = *bad ? __int_as_float(0x7fc00000) : sum;
    }
    ptx::cluster_sync();  // every CTA's sums are in its shared memory
    // CTA q writes columns [32 q, 32 q + 32) of each sequence: the SPLIT sums in rank order
    if (threadIdx.x < BCH * 32) {
      const int k = threadIdx.x >> 5, c = (int)q * 32 + (threadIdx.x & 31);
      const uint32_t src = ptx::smem_u32(ycta + k * 128 + c);
      float sum = ptx::ld_cluster_f32(ptx::map_to(src, 0));
#pragma unroll
      for (int rr = 1; rr < SPLIT; ++rr) sum += ptx::ld_cluster_f32(ptx::map_to(src, rr));
      if (k < nb && c < ncol) y[((int64_t)(b0 + k) * H + h) * V + v0 + c] = sum;
    }
    ptx::cluster_sync();  // the sums have been read before they are overwritten or freed
  }
  // the copies are complete before the CTA leaves (a copy that has not landed by
  // the first wait's limit gets one more bounded wait)
  if (warp == 0 && *bad) {
    for (int c = 0; c < NCHUNK; ++c) ptx::mbar_wait(&bars[c], 0, bad + 1, WUV_WAIT_NS);
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
      return cudaFuncSetAttribute(wuv_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  BULK_SMEM);
    }, &done);
    if (e != cudaSuccess) return e;
    wuv_bulk_kernel<<<dim3(H * SPLIT, (V + 127) / 128), BT, BULK_SMEM, s>>>(o, w, B, H, V, y);
  }
  else
    wuv_kernel<<<grid, WT, 0, s>>>(o, w, B, H, V, y);
  return cudaGetLastError();
}

}  // namespace kv8
