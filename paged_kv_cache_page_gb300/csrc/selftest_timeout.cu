// Test-only: the bounded pipeline wait of the attention kernels (mbar_wait
// in pa_common.cuh) on an mbarrier that no thread ever arrives at.  The wait
// gives up after its time limit, the kernel records PA_DEVERR_TIMEOUT in the
// error word and returns, and the CUDA context stays usable: the failure path
// is exercised without a fault, a trap or a hang.
#include "pa_common.cuh"

namespace pa {
namespace {

__global__ void wait_timeout_kernel(int32_t* err, unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 of a fresh barrier with one expected arrival never completes
    const unsigned long long t0 = globaltimer();
    if (!mbar_wait(&bar, 0)) report(err, PA_DEVERR_TIMEOUT, -1, 99);
    *elapsed_ns = globaltimer() - t0;
  }
}

}  // namespace
}  // namespace pa

extern "C" __attribute__((visibility("default"))) int pa_selftest_wait_timeout(
    int32_t* err, unsigned long long* elapsed_ns, cudaStream_t st) {
  pa::wait_timeout_kernel<<<1, 32, 0, st>>>(err, elapsed_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
