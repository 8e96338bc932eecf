// Self-test of the kernels' bounded waits (no paper counterpart).  Every wait of the
// tensor-core kernels on an mbarrier gives up after a time limit, records an error bit and
// lets the kernel leave instead of hanging the device.  This launch makes such a wait run out
// on purpose -- on a barrier that nothing arrives on -- so that the give-up path, the error
// bit and the device's continued use can be checked.  Nothing faults or traps: the wait ends
// by itself after the (clamped) limit.
#include "kda_internal.cuh"
#include "tc_prims.cuh"

namespace kda {
namespace {

__device__ unsigned int g_selftest_error;  // bit 3: the self-test's wait gave up (expected)

__global__ void bounded_wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one arrival expected; none is ever made
    tc::fence_mbar_init();
    if (!tc::mbar_wait(&bar, 0, limit_ns)) atomicOr(&g_selftest_error, 8u);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

unsigned int selftest_read_error(bool reset) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof(v));
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_selftest_error, &z, sizeof(z));
  }
  return v;
}

}  // namespace kda
