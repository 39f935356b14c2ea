// Diagnostic kernel: one bounded mbarrier wait that nothing ever completes,
// so the time-out path (status word + early return) can be exercised on a
// GPU without a fault or a hang.
#include "q6_internal.cuh"

namespace q6 {
namespace {

__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival; none is made
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, status, 0xEEu, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned int* status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace q6
