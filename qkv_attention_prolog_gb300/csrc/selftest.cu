// Self-test of the kernels' failure path: a bounded mbarrier wait that runs out.
//
// Every wait in the product kernels goes through mbar_wait (ptx.cuh): after kWaitLimitNs of
// %globaltimer it raises the CTA's abort flag and returns false, the kernel winds down and the
// workspace error word gets kErrTimeout, which mlap_check_errors reports as MLAP_ERR_TIMEOUT.
// This kernel runs that same wait on an mbarrier that nothing ever completes, so the path can
// be exercised on a GPU without faulting, trapping or hanging it: the wait ends by itself.
#include "ptx.cuh"
#include "internal.h"
#include "mlaprolog.h"

namespace mlap {

namespace {

__global__ void bounded_wait_kernel(uint32_t* __restrict__ err_word) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // no thread arrives on `bar`: phase 0 never completes and the wait gives up
    if (!mbar_wait(&bar, 0, &abort_flag)) atomicOr(err_word, kErrTimeout);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint32_t* err_word, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(err_word);
  return cudaGetLastError();
}

}  // namespace mlap
