// ablation.cu -- the fusion-level and incremental-form ablations of RedFuser
// (Figure 3: unfused vs fused cascades; Figure 4: non-incremental vs
// incremental computation; Figures 6-7: fusion at different levels), as
// alternative kernels for two cascades of this library.  They exist to be
// measured against the fused incremental kernels; they are correct but not
// tuned beyond plain 16-byte accesses.
//
// residual + LayerNorm (levels: mean, variance, normalise):
//   variant 1  fused, non-incremental: one CTA per row stages h = x + r in
//              shared memory (on-chip memory grows with the row), then a
//              mean pass, a variance pass and a normalise pass over it.
//   variant 2  fused up to level 2: one kernel computes (mean, rstd) per row,
//              a second kernel re-reads x and r to normalise.
//   variant 3  unfused: h to HBM, mean kernel, variance kernel, normalise
//              kernel; every level re-reads its input from HBM.
// softmax cross-entropy (levels: max, sum of exponentials, loss):
//   variant 1  fused, two passes: one CTA per row reads the row once for the
//              max, then again for the sum of exponentials (the second level
//              waits for the first to finish: no incremental rescale).
//   variant 2  unfused: a max kernel, a sum-of-exponentials kernel and a loss
//              kernel, each reading what it needs from HBM.
// (Variant 0, fused incremental, is the production kernel.)
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kT = 256;  // threads per CTA for the per-row kernels

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < blockDim.x / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = -INFINITY;
  for (int w = 0; w < blockDim.x / 32; ++w) t = fmaxf(t, red[w]);
  __syncthreads();
  return t;
}

// ------------------------------------------------------------------ LayerNorm
template <Dt DT>
__global__ void __launch_bounds__(kT) ln_smem_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                     const uint4* __restrict__ g, const uint4* __restrict__ b,
                                                     uint4* __restrict__ out, int nvec, float inv_cols, float eps) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  extern __shared__ float srow[];  // the whole row: cols floats
  __shared__ float red[32];
  const long long base = static_cast<long long>(blockIdx.x) * nvec;
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float xf[E], rf_[E];
    P::unpack(ld_stream(x + base + c), xf);
    P::unpack(ld_stream(r + base + c), rf_);
#pragma unroll
    for (int e = 0; e < E; ++e) srow[c * E + e] = xf[e] + rf_[e];
  }
  __syncthreads();
  const int cols = nvec * E;
  float s = 0.f;
  for (int i = threadIdx.x; i < cols; i += kT) s += srow[i];
  const float mean = block_sum(s, red) * inv_cols;  // level 1: needs the whole row
  float q = 0.f;
  for (int i = threadIdx.x; i < cols; i += kT) {
    const float d = srow[i] - mean;
    q = fmaf(d, d, q);
  }
  const float rstd = rsqrtf(block_sum(q, red) * inv_cols + eps);  // level 2: needs level 1
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float gf[E], bf[E], y[E];
    P::unpack(__ldg(g + c), gf);
    P::unpack(__ldg(b + c), bf);
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf((srow[c * E + e] - mean) * rstd, gf[e], bf[e]);
    st_stream(out + base + c, P::pack(y));
  }
}

// Reductions fused, normalise separate: (mean, rstd) of each row of x + r in
// one read, in the incremental form (each 16-byte block's own mean and sum of
// squared deviations are folded into the thread's running pair by the
// pairwise update of Chan et al.), then the same combine across the CTA.
struct Moments {
  float n, mean, m2;
};
__device__ __forceinline__ Moments moments_combine(Moments a, Moments b) {
  const float n = a.n + b.n;
  if (n == 0.f) return a;
  const float d = b.mean - a.mean, wb = b.n / n;
  return Moments{n, fmaf(d, wb, a.mean), a.m2 + b.m2 + d * d * a.n * wb};
}

template <Dt DT>
__global__ void __launch_bounds__(kT) ln_stats_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                      float2* __restrict__ stats, int nvec, float eps) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  __shared__ Moments red[32];
  const long long base = static_cast<long long>(blockIdx.x) * nvec;
  Moments run{0.f, 0.f, 0.f};
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float xf[E], rf_[E];
    P::unpack(ld_stream(x + base + c), xf);
    P::unpack(ld_stream(r + base + c), rf_);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      xf[e] += rf_[e];
      s += xf[e];
    }
    const float mb = s * (1.0f / E);
    float q = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) q = fmaf(xf[e] - mb, xf[e] - mb, q);
    run = moments_combine(run, Moments{static_cast<float>(E), mb, q});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Moments b{__shfl_xor_sync(0xffffffffu, run.n, o), __shfl_xor_sync(0xffffffffu, run.mean, o),
                    __shfl_xor_sync(0xffffffffu, run.m2, o)};
    run = moments_combine(run, b);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = run;
  __syncthreads();
  if (threadIdx.x == 0) {
    Moments t = red[0];
    for (int w = 1; w < kT / 32; ++w) t = moments_combine(t, red[w]);
    stats[blockIdx.x] = make_float2(t.mean, rsqrtf(t.m2 / t.n + eps));
  }
}

template <Dt DT>
__global__ void __launch_bounds__(kT) ln_apply_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                      const uint4* __restrict__ g, const uint4* __restrict__ b,
                                                      const float2* __restrict__ stats, uint4* __restrict__ out,
                                                      int nvec) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  const long long base = static_cast<long long>(blockIdx.x) * nvec;
  const float2 st = stats[blockIdx.x];
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float xf[E], rf_[E], gf[E], bf[E], y[E];
    P::unpack(ld_stream(x + base + c), xf);
    if (r) {
      P::unpack(ld_stream(r + base + c), rf_);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) rf_[e] = 0.f;
    }
    P::unpack(__ldg(g + c), gf);
    P::unpack(__ldg(b + c), bf);
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf((xf[e] + rf_[e] - st.x) * st.y, gf[e], bf[e]);
    st_stream(out + base + c, P::pack(y));
  }
}

// unfused pieces
template <Dt DT>
__global__ void add_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r, uint4* __restrict__ h,
                           long long nvec_total) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nvec_total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float a[E], c[E];
    P::unpack(ld_stream(x + i), a);
    P::unpack(ld_stream(r + i), c);
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] += c[e];
    st_stream(h + i, P::pack(a));
  }
}

template <Dt DT>
__global__ void __launch_bounds__(kT) row_mean_kernel(const uint4* __restrict__ h, float* __restrict__ mean,
                                                      int nvec, float inv_cols) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  __shared__ float red[32];
  const long long base = static_cast<long long>(blockIdx.x) * nvec;
  float s = 0.f;
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float a[E];
    P::unpack(ld_stream(h + base + c), a);
#pragma unroll
    for (int e = 0; e < E; ++e) s += a[e];
  }
  const float t = block_sum(s, red);
  if (threadIdx.x == 0) mean[blockIdx.x] = t * inv_cols;
}

template <Dt DT>
__global__ void __launch_bounds__(kT) row_rstd_kernel(const uint4* __restrict__ h, const float* __restrict__ mean,
                                                      float2* __restrict__ stats, int nvec, float inv_cols,
                                                      float eps) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  __shared__ float red[32];
  const long long base = static_cast<long long>(blockIdx.x) * nvec;
  const float mu = mean[blockIdx.x];
  float q = 0.f;
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float a[E];
    P::unpack(ld_stream(h + base + c), a);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float d = a[e] - mu;
      q = fmaf(d, d, q);
    }
  }
  const float t = block_sum(q, red);
  if (threadIdx.x == 0) stats[blockIdx.x] = make_float2(mu, rsqrtf(t * inv_cols + eps));
}

// ------------------------------------------------------------------ softmax cross-entropy
template <Dt DT>
__device__ __forceinline__ float xent_target_logit(const uint4* logits, long long row, long long V, long long t) {
  const uint16_t* z16 = reinterpret_cast<const uint16_t*>(logits);
  if constexpr (DT == Dt::F32) return reinterpret_cast<const float*>(logits)[row * V + t];
  else if constexpr (DT == Dt::BF16) return __uint_as_float(static_cast<uint32_t>(z16[row * V + t]) << 16);
  else return __half2float(__ushort_as_half(z16[row * V + t]));
}

template <Dt DT>
__device__ __forceinline__ float row_max_pass(const uint4* zr, int nvec, float* red) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  float m = -INFINITY;
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float z[E];
    P::unpack(ld_stream(zr + c), z);
#pragma unroll
    for (int e = 0; e < E; ++e) m = fmaxf(m, z[e]);
  }
  return block_max(m, red);
}

template <Dt DT>
__device__ __forceinline__ float row_sumexp_pass(const uint4* zr, int nvec, float m, float* red) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  float s = 0.f;
  for (int c = threadIdx.x; c < nvec; c += kT) {
    float z[E];
    P::unpack(ld_stream(zr + c), z);
#pragma unroll
    for (int e = 0; e < E; ++e) s += expf(z[e] - m);
  }
  return block_sum(s, red);
}

__device__ __forceinline__ float xent_loss(float lse, float zt, long long t, long long V, long long ignore) {
  if (t == ignore) return 0.f;
  if (t < 0 || t >= V) return __int_as_float(0x7fc00000);
  return lse - zt;
}

template <Dt DT>
__global__ void __launch_bounds__(kT) xent_twopass_kernel(const uint4* __restrict__ logits,
                                                          const long long* __restrict__ targets,
                                                          float* __restrict__ loss, float* __restrict__ lse_out,
                                                          int nvec, long long ignore) {
  __shared__ float red[32];
  const long long row = blockIdx.x;
  const uint4* zr = logits + row * nvec;
  const float m = row_max_pass<DT>(zr, nvec, red);        // level 1 over the whole row first
  const float s = row_sumexp_pass<DT>(zr, nvec, m, red);  // level 2 re-reads the row
  if (threadIdx.x == 0) {
    const float lse = m + logf(s);
    const long long V = static_cast<long long>(nvec) * Pack<DT>::E, t = targets[row];
    const bool in_range = t >= 0 && t < V;
    if (lse_out) lse_out[row] = lse;
    loss[row] = xent_loss(lse, in_range ? xent_target_logit<DT>(logits, row, V, t) : 0.f, t, V, ignore);
  }
}

template <Dt DT>
__global__ void __launch_bounds__(kT) xent_max_kernel(const uint4* __restrict__ logits, float* __restrict__ mx,
                                                      int nvec) {
  __shared__ float red[32];
  const float m = row_max_pass<DT>(logits + static_cast<long long>(blockIdx.x) * nvec, nvec, red);
  if (threadIdx.x == 0) mx[blockIdx.x] = m;
}

template <Dt DT>
__global__ void __launch_bounds__(kT) xent_lse_kernel(const uint4* __restrict__ logits, const float* __restrict__ mx,
                                                      float* __restrict__ lse, int nvec) {
  __shared__ float red[32];
  const float m = mx[blockIdx.x];
  const float s = row_sumexp_pass<DT>(logits + static_cast<long long>(blockIdx.x) * nvec, nvec, m, red);
  if (threadIdx.x == 0) lse[blockIdx.x] = m + logf(s);
}

template <Dt DT>
__global__ void xent_loss_kernel(const uint4* __restrict__ logits, const long long* __restrict__ targets,
                                 const float* __restrict__ lse, float* __restrict__ loss, float* __restrict__ lse_out,
                                 int rows, long long V, long long ignore) {
  const long long row = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (row >= rows) return;
  const long long t = targets[row];
  const bool in_range = t >= 0 && t < V;
  if (lse_out) lse_out[row] = lse[row];
  loss[row] = xent_loss(lse[row], in_range ? xent_target_logit<DT>(logits, row, V, t) : 0.f, t, V, ignore);
}

template <Dt DT>
cudaError_t ln_variant(const void* x, const void* r, const void* g, const void* b, void* out, int rows, int cols,
                       float eps, int variant, void* ws, cudaStream_t s) {
  constexpr int E = Pack<DT>::E;
  const int nvec = cols / E;
  const float inv = 1.0f / static_cast<float>(cols);
  auto X = static_cast<const uint4*>(x);
  auto R = static_cast<const uint4*>(r);
  auto G = static_cast<const uint4*>(g);
  auto Bt = static_cast<const uint4*>(b);
  auto O = static_cast<uint4*>(out);
  if (variant == 1) {
    const size_t smem = static_cast<size_t>(cols) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(ln_smem_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    ln_smem_kernel<DT><<<rows, kT, smem, s>>>(X, R, G, Bt, O, nvec, inv, eps);
  } else if (variant == 2) {
    auto st = static_cast<float2*>(ws);
    ln_stats_kernel<DT><<<rows, kT, 0, s>>>(X, R, st, nvec, eps);
    ln_apply_kernel<DT><<<rows, kT, 0, s>>>(X, R, G, Bt, st, O, nvec);
  } else {
    auto st = static_cast<float2*>(ws);
    auto mean = reinterpret_cast<float*>(st + rows);
    auto h = reinterpret_cast<uint4*>(static_cast<char*>(ws) + ((static_cast<size_t>(rows) * 12 + 255) & ~size_t(255)));
    add_kernel<DT><<<1216, 256, 0, s>>>(X, R, h, static_cast<long long>(rows) * nvec);
    row_mean_kernel<DT><<<rows, kT, 0, s>>>(h, mean, nvec, inv);
    row_rstd_kernel<DT><<<rows, kT, 0, s>>>(h, mean, st, nvec, inv, eps);
    ln_apply_kernel<DT><<<rows, kT, 0, s>>>(h, nullptr, G, Bt, st, O, nvec);
  }
  return cudaGetLastError();
}

template <Dt DT>
cudaError_t xent_variant(const void* logits, const long long* targets, float* loss, float* lse, int rows, int vocab,
                         long long ignore, int variant, void* ws, cudaStream_t s) {
  constexpr int E = Pack<DT>::E;
  const int nvec = vocab / E;
  auto L = static_cast<const uint4*>(logits);
  if (variant == 1) {
    xent_twopass_kernel<DT><<<rows, kT, 0, s>>>(L, targets, loss, lse, nvec, ignore);
  } else {
    auto mx = static_cast<float*>(ws);
    auto l2 = mx + rows;
    xent_max_kernel<DT><<<rows, kT, 0, s>>>(L, mx, nvec);
    xent_lse_kernel<DT><<<rows, kT, 0, s>>>(L, mx, l2, nvec);
    xent_loss_kernel<DT><<<(rows + 255) / 256, 256, 0, s>>>(L, targets, l2, loss, lse, rows, vocab, ignore);
  }
  return cudaGetLastError();
}

}  // namespace

size_t ablation_ln_workspace_bytes(int rows, int cols, int variant, Dt dt) {
  if (variant == 2) return static_cast<size_t>(rows) * 8;
  if (variant == 3)
    return ((static_cast<size_t>(rows) * 12 + 255) & ~size_t(255)) +
           static_cast<size_t>(rows) * cols * (dt == Dt::F32 ? 4 : 2);
  return 0;
}

size_t ablation_xent_workspace_bytes(int rows, int variant) {
  return variant == 2 ? static_cast<size_t>(rows) * 8 : 0;
}

cudaError_t launch_ln_ablation(const void* x, const void* r, const void* g, const void* b, void* out, int rows,
                               int cols, float eps, int variant, void* ws, Dt dt, cudaStream_t s) {
  switch (dt) {
    case Dt::F32: return ln_variant<Dt::F32>(x, r, g, b, out, rows, cols, eps, variant, ws, s);
    case Dt::F16: return ln_variant<Dt::F16>(x, r, g, b, out, rows, cols, eps, variant, ws, s);
    case Dt::BF16: return ln_variant<Dt::BF16>(x, r, g, b, out, rows, cols, eps, variant, ws, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_xent_ablation(const void* logits, const long long* targets, float* loss, float* lse, int rows,
                                 int vocab, long long ignore, int variant, void* ws, Dt dt, cudaStream_t s) {
  switch (dt) {
    case Dt::F32: return xent_variant<Dt::F32>(logits, targets, loss, lse, rows, vocab, ignore, variant, ws, s);
    case Dt::F16: return xent_variant<Dt::F16>(logits, targets, loss, lse, rows, vocab, ignore, variant, ws, s);
    case Dt::BF16: return xent_variant<Dt::BF16>(logits, targets, loss, lse, rows, vocab, ignore, variant, ws, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rf
