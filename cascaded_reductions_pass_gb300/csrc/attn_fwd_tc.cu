// attn_fwd_tc.cu -- placeholder until the tcgen05 attention kernel lands.
#include "rf_device.cuh"
namespace rf {
cudaError_t launch_attn_tc(const void*, const void*, const void*, void*, float*, int, int, int, int, int, int,
                           float, int, Dt, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace rf
