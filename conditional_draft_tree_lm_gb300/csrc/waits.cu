// Self-check of the bounded waits every kernel relies on: a grid barrier that
// one participant never reaches, and an mbarrier phase that nothing completes.
// Both give up after the wait limit, record DT_DEV_TIMEOUT in the status word
// and return, so the context stays usable; nothing faults, traps or hangs.
#include "chainlib.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dt {

namespace {

// which = 0: a grid barrier of two CTAs where CTA 1 leaves without arriving;
// which = 1: one CTA waits on an mbarrier that no thread arrives on.
__global__ void __launch_bounds__(cl::kThreads, 1) k_wait_check(unsigned* bar, int* status, int which) {
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_mbar;
  if (which == 0) {
    if (blockIdx.x != 0) return;  // the missing participant
    unsigned epoch = 0;
    cl::grid_barrier(bar, epoch, status, &s_abort);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&s_mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&s_mbar, 0u, status);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_check(unsigned* bar, int* status, int which, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(which == 0 ? 2 : 1);
  cfg.blockDim = dim3(cl::kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = which == 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_wait_check, bar, status, which);
}

}  // namespace dt
