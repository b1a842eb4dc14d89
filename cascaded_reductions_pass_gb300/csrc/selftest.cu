// selftest.cu -- exercises the failure paths on the GPU without hanging or
// faulting it.  The bounded-wait path: one warp waits on an mbarrier that nothing arrives
// on, gives up after a short limit, records RF_ERR_TIMEOUT in the device
// status word exactly as the production kernels do, and returns.  Nothing is
// in flight (no TMA copy, no tensor-memory allocation) when it gives up.
// The index-check path of RF_CHECKS builds: one thread evaluates a check that
// fails, with no memory access behind it.
#include "rf_device.cuh"

namespace rf {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, unsigned* status, int* waited_out) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_for(&bar, 0, limit_ns));
  if (!ok && threadIdx.x == 0) {
    atomicOr(status, kStatusTimeout);
    if (waited_out) *waited_out = 1;
  }
}

// An index that lies past a (phantom) buffer of 8 elements: the check fails
// and, in a checked build, records kStatusCheck; no access is made either way.
__global__ void __launch_bounds__(32) check_kernel(unsigned* status, int idx) {
  if (threadIdx.x == 0) (void)RF_INB(idx < 8, status);
}

}  // namespace

cudaError_t launch_check_selftest(unsigned* status, cudaStream_t s) {
  check_kernel<<<1, 32, 0, s>>>(status, 8);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned* status, int* waited_out, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status, waited_out);
  return cudaGetLastError();
}

}  // namespace rf
