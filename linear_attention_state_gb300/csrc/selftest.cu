// Self-test of the bounded-wait path every tensor-core kernel relies on: one thread waits
// on an mbarrier that nothing ever arrives at, with the caller's cycle limit, records
// HYPIC_ETIMEOUT in the status word and returns.  Nothing faults and nothing hangs.
#include "tc_ptx.cuh"

namespace hypic {
namespace {

__global__ void bounded_wait_kernel(long long limit_cycles, int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait_cycles(&bar, 0, err, limit_cycles);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(long long limit_cycles, int *err, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>(limit_cycles, err);
  return cudaGetLastError();
}

}  // namespace hypic
