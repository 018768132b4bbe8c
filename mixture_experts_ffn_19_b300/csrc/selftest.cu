// The device-side failure paths, exercised without a fault.
//
// (1) One CTA waits on an mbarrier that nothing arrives on, through the same
// bounded wait every pipeline role uses (mbar_wait), with a short limit.  When
// the limit runs out the wait records the time-out in the workspace status
// word and the kernel returns, exactly as a stalled GEMM or router pipeline
// would; the context stays usable.
//
// (2) A cooperative grid in which CTA 0, by construction, never reaches the
// grid barrier (the same grid_barrier the reroute kernel uses) while the other
// CTAs run a chain of barriers.  Their first wait runs out, the first CTA to
// give up records the time-out and raises the abort flag, and every CTA leaves
// the chain at once: a stalled grid costs one limit, not one per barrier.
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

__global__ void barrier_selftest_kernel(GridBarrier* bar, int* status, uint64_t limit_ns,
                                        int n_barriers) {
  if (blockIdx.x == 0) return;                   // never arrives
  for (int i = 0; i < n_barriers; ++i)
    if (!grid_barrier(bar, status, limit_ns)) return;
  // every barrier passed: CTA 0 would have had to arrive, which it never does
  if (threadIdx.x == 0) set_status(status, kDevBadState);
}

}  // namespace

cudaError_t launch_barrier_selftest(int* status, GridBarrier* bar, uint64_t limit_ns,
                                    int n_barriers, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(bar, 0, sizeof(GridBarrier), s);
  if (err != cudaSuccess) return err;
  GridBarrier* b = bar;
  int* st = status;
  uint64_t lim = limit_ns;
  int nb = n_barriers;
  void* args[] = {&b, &st, &lim, &nb};
  // four CTAs of one warp: co-resident on any device, as a cooperative launch requires
  err = cudaLaunchCooperativeKernel((const void*)barrier_selftest_kernel, dim3(4), dim3(32),
                                    args, 0, s);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
