// selftest.cu -- a bounded wait that nothing completes, for testing the
// timeout path of the pipelines' waits without faulting or hanging the GPU.
//
// One thread initialises an mbarrier that expects one arrival which never
// comes and waits on it through mbar_wait, the helper every pipeline wait of
// the library uses; the wait gives up after the context's wait limit, records
// MOE_ERR_TIMEOUT on the error word and the kernel returns.  The thread then
// arrives on the barrier itself so that its phase completes before the CTA
// leaves.
#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void wait_selftest_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const bool done = mbar_wait(&bar, 0, err);  // no one arrives: runs out after the limit
  if (!done) mbar_arrive(&bar);
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, cudaStream_t s) {
  return launch("wait_selftest", wait_selftest_kernel, dim3(1), dim3(32), 0, s, false, err);
}

}  // namespace moe
