// Diagnostic kernel for the bounded-wait machinery every tcgen05 kernel of
// this library uses: one thread waits on an mbarrier that nothing
// completes, with a short limit; the wait gives up and the CTA records a
// timeout in the status word instead of hanging or trapping.
#include "tc_ptx.cuh"
#include "usp_common.cuh"

namespace {

__global__ void bounded_wait_kernel(uint64_t limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);   // expects one arrival that never comes
    abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!tc::mbar_wait(&bar, 0, &abort, limit_ns)) usp::set_status(status, usp::kErrTimeout);
  }
}

}  // namespace

cudaError_t usp_launch_bounded_wait(int64_t limit_ns, unsigned* status, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>((uint64_t)limit_ns, status);
  usp_count_launches(1);
  return cudaGetLastError();
}
