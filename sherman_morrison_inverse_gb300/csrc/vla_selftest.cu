// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing
// completes, gives up after the limit and reports a timeout in the status block,
// exactly as a scan kernel does when an input copy or a tensor-core product never
// lands.  Nothing faults and nothing hangs; the context stays usable.
#include "vla_internal.cuh"

namespace vla {
namespace {

__global__ void wait_selftest_kernel(DevStatus* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival expected; none ever comes
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, limit_ns)) atomicOr(&status->flags, kStatusTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(DevStatus* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace vla
