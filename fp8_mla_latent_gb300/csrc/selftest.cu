// selftest.cu -- a check of the kernels' failure path without a GPU fault: one
// warp waits, through the same bounded mbarrier wait the decode kernels use, on
// a barrier that nothing arrives at.  The wait gives up after the given limit,
// the error word records a timeout, and the kernel returns normally, so the
// context stays usable.
#include "kv8_common.cuh"
#include "tc_ptx.cuh"

namespace kv8 {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // phase 0 never completes: nothing arrives on the barrier
  const bool ok = ptx::mbar_wait_warp(&bar, 0, &abort_flag, limit_ns);
  if (!ok && threadIdx.x == 0) atomicOr(err, ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout(unsigned* err, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace kv8
