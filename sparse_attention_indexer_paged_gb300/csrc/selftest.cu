// Self-test of the failure path every kernel of the library shares: a
// pipeline wait that sees no progress gives up after its time limit, records
// DSA_ERR_TIMEOUT in the caller's status word and returns, leaving the
// context usable.  Here the wait is on an mbarrier that nothing arrives on.
#include "ptx.cuh"

namespace dsa {
namespace {

__global__ void selftest_wait_kernel(uint64_t timeout_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_word;
  volatile int32_t* abort_flag = &abort_word;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);  // one arrival would complete phase 0; none comes
  *abort_flag = 0;
  fence_mbar_init();
  wait_or_abort_for(b, 0, abort_flag, status, timeout_ns);  // runs out: reports DSA_ERR_TIMEOUT
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t timeout_ns, int32_t* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace dsa
