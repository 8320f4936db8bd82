// Self-test of the bounded mbarrier wait that guards every pipeline stage of the library's
// kernels: one thread waits on a phase that nothing completes, the wait runs out after its
// limit, records the timeout in the status words and returns, and the kernel exits
// normally, so the host sees L3_ERR_TIMEOUT with the device still usable.
#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {

namespace {

constexpr int kSelftestCode = 0x40000000;  // timeout bit of this test (no kernel uses it)

__global__ void wait_selftest_kernel(DevStatus* st, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  abort = 0;
  tc::fence_barrier_init();
  volatile int* flag = &abort;
  // phase 0 never completes: nothing arrives on the barrier
  tc::mbar_wait(&bar, 0, flag, st, kSelftestCode, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(DevStatus* st, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(st, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
