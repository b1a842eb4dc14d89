// lse_merge.cuh -- the log-sum-exp merge of partial attention results, as a
// kernel template shared by the merge entry point (lse_merge.cu) and the
// split tail of the tensor-core attention forward (attn_fwd_tc.cu).
//
// Each part s carries its normalised output O_s and its lse_s = m_s + ln l_s.
// The whole key set's level-2 sum is sum_s exp(lse_s), so LSE = ln of it, and
// its level-3 result is O = sum_s exp(lse_s - LSE) * O_s: the correction of
// each part's running result by one combine step (RedFuser, Table 1: reduce
// op + with combine op *; Figure 4, incremental form; Figure 13, the
// FlashDecoding IR whose split results this merges).  The log-sum-exp is taken
// relative to mx = max_s lse_s so that no exponential overflows, and each
// weight is formed as exp(lse_s - mx) / sum_s' exp(lse_s' - mx): mx is one of
// the inputs, so lse_s - mx is exact or nearly so.  exp(lse_s - LSE) would
// instead carry the rounding of LSE = mx + ln(sum), which is of the order of
// ulp(LSE) (3e-5 at LSE ~ 500), into every weight as a relative error.
//
// A part whose lse_s is NaN (a split kernel that gave up after a bounded wait
// marks its partials that way) makes the merged row NaN, so a result built
// from missing partials cannot pass for a valid one.
//
// One warp per row: lanes first reduce the parts' LSEs (max, then the sum of
// exponentials), write the S weights to shared memory, then each lane owns
// D/4/32 float4 columns of the output and sums the weighted parts.  Partials
// are [rows, S, D] and [rows, S] fp32; RowMap gives the output row of each
// partial row (a negative value skips the row).
#pragma once

#include <math.h>

#include "rf_device.cuh"

namespace rf {

struct IdentityRows {
  __device__ __forceinline__ long long operator()(long long r) const { return r; }
};

constexpr int kMergeWarps = 8;
constexpr int kMergeMaxSplits = 256;

template <Dt DT>
__device__ __forceinline__ void merge_store4(void* o, long long idx4, float4 v) {
  if constexpr (DT == Dt::F32) {
    reinterpret_cast<float4*>(o)[idx4] = v;
  } else {
    uint2 p;
    if constexpr (DT == Dt::BF16) {
      p.x = pack_bf16x2(v.x, v.y);
      p.y = pack_bf16x2(v.z, v.w);
    } else {
      p.x = pack_f16x2(v.x, v.y);
      p.y = pack_f16x2(v.z, v.w);
    }
    reinterpret_cast<uint2*>(o)[idx4] = p;
  }
}

template <Dt DT, class RowMap>
__global__ void __launch_bounds__(kMergeWarps * 32) lse_merge_kernel(const float* __restrict__ o_part,
                                                                     const float* __restrict__ lse_part,
                                                                     void* __restrict__ o, float* __restrict__ lse,
                                                                     int rows, int S, int D, RowMap out_row,
                                                                     long long out_rows, unsigned* status) {
  __shared__ float s_w[kMergeWarps][kMergeMaxSplits];
  griddep_wait();  // the kernel that wrote the partials has completed (after the attention split tail and the
                   // split-KV decode this kernel is launched early; otherwise this returns at once)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
  if (row >= rows) return;
  const long long orow = out_row(row);  // where this row's result goes (< 0: nowhere)
  if (orow < 0 || !RF_INB(orow < out_rows && S <= kMergeMaxSplits, status)) return;
  const float* lp = lse_part + row * S;

  float mx = -INFINITY;
  bool bad = false;
  for (int s = lane; s < S; s += 32) {
    const float v = lp[s];
    bad |= v != v;
    mx = fmaxf(mx, v);
  }
  mx = warp_max(mx);
  const int D4 = D >> 2;
  if (__any_sync(0xffffffffu, bad)) {  // a part is marked invalid
    for (int j = lane; j < D4; j += 32) merge_store4<DT>(o, orow * D4 + j, make_float4(NAN, NAN, NAN, NAN));
    if (lse && lane == 0) lse[orow] = NAN;
    return;
  }
  if (mx == -INFINITY) {  // every part empty
    for (int j = lane; j < D4; j += 32) merge_store4<DT>(o, orow * D4 + j, make_float4(0.f, 0.f, 0.f, 0.f));
    if (lse && lane == 0) lse[orow] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int s = lane; s < S; s += 32) sum += expf(lp[s] - mx);
  sum = warp_sum(sum);
  const float L = mx + logf(sum);
  for (int s = lane; s < S; s += 32) s_w[warp][s] = expf(lp[s] - mx) / sum;
  __syncwarp();
  if (lse && lane == 0) lse[orow] = L;

  const float4* op = reinterpret_cast<const float4*>(o_part) + row * S * D4;
  for (int j = lane; j < D4; j += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= S; s += 4) {
      float4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = __ldg(op + (s + u) * D4 + j);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w = s_w[warp][s + u];
        acc.x = fmaf(w, a[u].x, acc.x);
        acc.y = fmaf(w, a[u].y, acc.y);
        acc.z = fmaf(w, a[u].z, acc.z);
        acc.w = fmaf(w, a[u].w, acc.w);
      }
    }
    for (; s < S; ++s) {
      const float4 a = __ldg(op + s * D4 + j);
      const float w = s_w[warp][s];
      acc.x = fmaf(w, a.x, acc.x);
      acc.y = fmaf(w, a.y, acc.y);
      acc.z = fmaf(w, a.z, acc.z);
      acc.w = fmaf(w, a.w, acc.w);
    }
    merge_store4<DT>(o, orow * D4 + j, acc);
  }
}

}  // namespace rf
