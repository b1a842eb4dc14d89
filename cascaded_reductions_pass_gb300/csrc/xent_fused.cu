// xent_fused.cu -- fused softmax + cross-entropy over vocabulary-sized rows.
//
// The loss of one row is a cascade of the same form as attention's safe
// softmax ("Operator Fusion" guide, section 3, lists softmax + cross-entropy as
// fusible): level 1 the row max m (reduce max, combine +), level 2
// l = sum_j exp(z_j - m) (reduce +, combine *), then loss = m + ln l - z_t.
// It runs in the incremental form of RedFuser's Figure 4: each thread keeps a
// running (m, l) and, when a 16-byte block raises m, rescales l by
// exp(m_old - m_new) before adding the block.  The threads of the row are then
// merged with the same log-sum-exp combine (warp shuffles, then shared
// memory), so the logits are read from HBM once.  The optional gradient
// softmax(z) - onehot(t) is a second pass over the row, which the CTA has just
// read and which is normally still in L2.
//
// One CTA of 512 threads per row; each thread keeps four 16-byte loads in
// flight.  The vocabulary must be a multiple of one 16-byte vector.
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// (m, l) with m in base-2 units (z * log2 e) and l = sum 2^(x - m).
struct Run {
  float m, l;
};

__device__ __forceinline__ Run lse_combine(Run a, Run b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return Run{-INFINITY, 0.f};
  return Run{M, a.l * ex2_ftz(a.m - M) + b.l * ex2_ftz(b.m - M)};
}

template <Dt DT>
__device__ __forceinline__ void fold_block(const uint4& u, Run& r) {
  constexpr int E = Pack<DT>::E;
  float z[E];
  Pack<DT>::unpack(u, z);
  float bm = z[0];
#pragma unroll
  for (int e = 1; e < E; ++e) bm = fmaxf(bm, z[e]);
  bm *= kLog2e;
  if (bm > r.m) {  // level 1 moved: correct level 2 by 2^(m_old - m_new)
    r.l *= ex2_ftz(r.m - bm);
    r.m = bm;
  }
  if (r.m == -INFINITY) return;  // nothing finite seen yet (all -inf logits)
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s += ex2_ftz(fmaf(z[e], kLog2e, -r.m));
  r.l += s;
}

template <Dt DT>
__global__ void __launch_bounds__(kThreads) xent_kernel(const uint4* __restrict__ logits,
                                                        const long long* __restrict__ targets,
                                                        float* __restrict__ loss, float* __restrict__ lse_out,
                                                        uint4* __restrict__ grad, int nvec, long long ignore_index) {
  constexpr int E = Pack<DT>::E;
  __shared__ Run s_run[kThreads / 32];
  const long long row = blockIdx.x;
  const uint4* zr = logits + row * nvec;
  const int tid = threadIdx.x;

  Run run{-INFINITY, 0.f};
  int c = tid;
  for (; c + (kUnroll - 1) * kThreads < nvec; c += kUnroll * kThreads) {
    uint4 u[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) u[k] = ld_stream(zr + c + k * kThreads);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) fold_block<DT>(u[k], run);
  }
  for (; c < nvec; c += kThreads) fold_block<DT>(ld_stream(zr + c), run);

  // merge the row's threads: warp shuffles, then the warps in shared memory
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Run b{__shfl_xor_sync(0xffffffffu, run.m, o), __shfl_xor_sync(0xffffffffu, run.l, o)};
    run = lse_combine(run, b);
  }
  if ((tid & 31) == 0) s_run[tid >> 5] = run;
  __syncthreads();
  run = s_run[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) run = lse_combine(run, s_run[w]);
  const float lse2 = run.m + log2f(run.l);  // base 2
  const float lse = lse2 * kLn2;

  const long long t = targets[row];
  const long long V = static_cast<long long>(nvec) * E;
  const bool ignored = t == ignore_index;
  const bool in_range = t >= 0 && t < V;
  if (tid == 0) {
    if (lse_out) lse_out[row] = lse;
    float l = 0.f;
    if (!ignored) {
      if (in_range) {
        const uint16_t* z16 = reinterpret_cast<const uint16_t*>(logits);
        float zt;
        if constexpr (DT == Dt::F32)
          zt = reinterpret_cast<const float*>(logits)[row * V + t];
        else if constexpr (DT == Dt::BF16)
          zt = __uint_as_float(static_cast<uint32_t>(z16[row * V + t]) << 16);
        else
          zt = __half2float(__ushort_as_half(z16[row * V + t]));
        l = lse - zt;
      } else {
        l = __int_as_float(0x7fc00000);  // out-of-range target: NaN loss
      }
    }
    loss[row] = l;
  }
  if (grad == nullptr) return;

  // gradient pass: softmax(z) - onehot(t), or 0 for an ignored row
  uint4* gr = grad + row * nvec;
  for (int cc = tid; cc < nvec; cc += kThreads) {
    float g[E];
    if (ignored) {
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = 0.f;
    } else {
      float z[E];
      Pack<DT>::unpack(__ldg(zr + cc), z);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        g[e] = ex2_ftz(fmaf(z[e], kLog2e, -lse2));
        if (static_cast<long long>(cc) * E + e == t) g[e] -= 1.f;
      }
    }
    st_stream(gr + cc, Pack<DT>::pack(g));
  }
}

}  // namespace

cudaError_t launch_xent(const void* logits, const long long* targets, float* loss, float* lse, void* grad, int rows,
                        int vocab, long long ignore_index, Dt dt, cudaStream_t s) {
  const int E = dt == Dt::F32 ? 4 : 8;
  const int nvec = vocab / E;
  auto L = static_cast<const uint4*>(logits);
  auto G = static_cast<uint4*>(grad);
  switch (dt) {
    case Dt::F32: xent_kernel<Dt::F32><<<rows, kThreads, 0, s>>>(L, targets, loss, lse, G, nvec, ignore_index); break;
    case Dt::F16: xent_kernel<Dt::F16><<<rows, kThreads, 0, s>>>(L, targets, loss, lse, G, nvec, ignore_index); break;
    case Dt::BF16: xent_kernel<Dt::BF16><<<rows, kThreads, 0, s>>>(L, targets, loss, lse, G, nvec, ignore_index); break;
  }
  return cudaGetLastError();
}

}  // namespace rf
