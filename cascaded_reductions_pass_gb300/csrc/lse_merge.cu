// lse_merge.cu -- combine attention results computed over disjoint key sets.
//
// Each part s carries its normalised output O_s and its lse_s = m_s + ln l_s.
// The whole key set's level-2 sum is sum_s exp(lse_s), so LSE = ln of it, and
// its level-3 result is O = sum_s exp(lse_s - LSE) * O_s: the correction of
// each part's running result by one combine step (RedFuser, Table 1: reduce
// op + with combine op *; Figure 4, incremental form; Figure 13, the
// FlashDecoding IR whose split results this merges).  The log-sum-exp is taken
// relative to max_s lse_s so that no exponential overflows.
//
// One warp per row: lanes first reduce the parts' LSEs (max, then the sum of
// exponentials), write the S weights to shared memory, then each lane owns
// D/4/32 float4 columns of the output and sums the weighted parts.
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxSplits = 256;

template <Dt DT>
__device__ __forceinline__ void store4(void* o, long long idx4, float4 v) {
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

template <Dt DT>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const float* __restrict__ o_part,
                                                                const float* __restrict__ lse_part,
                                                                void* __restrict__ o, float* __restrict__ lse,
                                                                int rows, int S, int D) {
  __shared__ float s_w[kWarps][kMaxSplits];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + warp;
  if (row >= rows) return;
  const float* lp = lse_part + row * S;

  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[s]);
  mx = warp_max(mx);
  const int D4 = D >> 2;
  if (mx == -INFINITY) {  // every part empty
    for (int j = lane; j < D4; j += 32) store4<DT>(o, row * D4 + j, make_float4(0.f, 0.f, 0.f, 0.f));
    if (lse && lane == 0) lse[row] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int s = lane; s < S; s += 32) sum += expf(lp[s] - mx);
  sum = warp_sum(sum);
  const float L = mx + logf(sum);
  for (int s = lane; s < S; s += 32) s_w[warp][s] = expf(lp[s] - L);
  __syncwarp();
  if (lse && lane == 0) lse[row] = L;

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
    store4<DT>(o, row * D4 + j, acc);
  }
}

}  // namespace

cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int rows,
                             int splits, int D, Dt out_dt, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((static_cast<long long>(rows) + kWarps - 1) / kWarps);
  switch (out_dt) {
    case Dt::F32: lse_merge_kernel<Dt::F32><<<grid, kWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D); break;
    case Dt::F16: lse_merge_kernel<Dt::F16><<<grid, kWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D); break;
    case Dt::BF16: lse_merge_kernel<Dt::BF16><<<grid, kWarps * 32, 0, s>>>(o_part, lse_part, o, lse, rows, splits, D); break;
  }
  return cudaGetLastError();
}

}  // namespace rf
