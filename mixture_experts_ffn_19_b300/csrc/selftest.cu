// The device-side failure path, exercised without a fault: one CTA waits on an
// mbarrier that nothing arrives on, through the same bounded wait every
// pipeline role uses (mbar_wait), with a short limit.  When the limit runs
// out the wait records the time-out in the workspace status word and the
// kernel returns, exactly as a stalled GEMM or router pipeline would; the
// context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // every thread waits; nothing ever arrives, so each wait gives up
  mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
