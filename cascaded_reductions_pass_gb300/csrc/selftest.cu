// selftest.cu -- exercises the bounded-wait failure path on the GPU without
// hanging or faulting it: one warp waits on an mbarrier that nothing arrives
// on, gives up after a short limit, records RF_ERR_TIMEOUT in the device
// status word exactly as the production kernels do, and returns.  Nothing is
// in flight (no TMA copy, no tensor-memory allocation) when it gives up.
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

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned* status, int* waited_out, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status, waited_out);
  return cudaGetLastError();
}

}  // namespace rf
