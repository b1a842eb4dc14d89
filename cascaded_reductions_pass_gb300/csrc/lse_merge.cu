// lse_merge.cu -- combine attention results computed over disjoint key sets
// (the kernel is in lse_merge.cuh; this file launches it with output rows
// equal to partial rows).
#include "lse_merge.cuh"

namespace rf {

cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int rows,
                             int splits, int D, Dt out_dt, unsigned* status, cudaStream_t s, bool after_split) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>((static_cast<long long>(rows) + kMergeWarps - 1) / kMergeWarps));
  lc.blockDim = dim3(kMergeWarps * 32);
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = after_split ? 1 : 0;
  lc.attrs = la;
  lc.numAttrs = 1;
  const IdentityRows id;
  const long long out_rows = rows;
  switch (out_dt) {
    case Dt::F32:
      return cudaLaunchKernelEx(&lc, lse_merge_kernel<Dt::F32, IdentityRows>, o_part, lse_part, o, lse, rows, splits,
                                D, id, out_rows, status);
    case Dt::F16:
      return cudaLaunchKernelEx(&lc, lse_merge_kernel<Dt::F16, IdentityRows>, o_part, lse_part, o, lse, rows, splits,
                                D, id, out_rows, status);
    case Dt::BF16:
      return cudaLaunchKernelEx(&lc, lse_merge_kernel<Dt::BF16, IdentityRows>, o_part, lse_part, o, lse, rows,
                                splits, D, id, out_rows, status);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rf
