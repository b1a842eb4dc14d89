// lse_merge.cu -- combine attention results computed over disjoint key sets
// (the kernel is in lse_merge.cuh; this file launches it with output rows
// equal to partial rows).
#include "lse_merge.cuh"

namespace rf {

cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int rows,
                             int splits, int D, Dt out_dt, unsigned* status, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((static_cast<long long>(rows) + kMergeWarps - 1) / kMergeWarps);
  const IdentityRows id;
  switch (out_dt) {
    case Dt::F32: lse_merge_kernel<Dt::F32><<<grid, kMergeWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D, id, rows, status); break;
    case Dt::F16: lse_merge_kernel<Dt::F16><<<grid, kMergeWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D, id, rows, status); break;
    case Dt::BF16: lse_merge_kernel<Dt::BF16><<<grid, kMergeWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D, id, rows, status); break;
  }
  return cudaGetLastError();
}

}  // namespace rf
