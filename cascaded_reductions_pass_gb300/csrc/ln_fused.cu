// ln_fused.cu -- one-pass residual + LayerNorm ("Operator Fusion" guide,
// section 1 traffic example and section 2 Pattern 2: mean -> variance ->
// normalise; section 4 places eps inside the square root).
//
// The cascade mean -> M2 -> normalise runs in the incremental form of
// RedFuser (Figure 4): each thread keeps a running (count, mean, M2) that it
// updates as each 16-byte block of the row arrives (Chan, Golub and LeVeque's
// pairwise combine: the M2 of the union is M2_a + M2_b + delta^2 n_a n_b / n,
// the additive correction of level 2 when level 1 moves).  The same combine
// merges the threads of a row through warp shuffles and then across warps in
// shared memory.  The row stays in registers between the statistics and the
// normalisation, so x and the residual are read from HBM once and y is
// written once.
//
// Layout: a group of `tpr` threads (a multiple of 32) owns one row; thread t
// holds the row's 16-byte vectors t, t + tpr, ..., t + (VPT-1)*tpr.  A CTA
// holds max(1, 256 / tpr) rows.
#include "rf_device.cuh"

namespace rf {
namespace {

struct Stats {
  float n, mean, m2;
};

__device__ __forceinline__ Stats chan(Stats a, Stats b) {
  if (b.n == 0.f) return a;
  if (a.n == 0.f) return b;
  const float n = a.n + b.n;
  const float f = b.n / n;
  const float d = b.mean - a.mean;
  return Stats{n, fmaf(d, f, a.mean), a.m2 + b.m2 + d * d * a.n * f};
}

template <Dt DT, int VPT>
__global__ void __launch_bounds__(1024) ln_fused_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                        const uint4* __restrict__ gamma,
                                                        const uint4* __restrict__ beta, uint4* __restrict__ out,
                                                        uint4* __restrict__ r_out, int rows, int nvec, int tpr,
                                                        float inv_cols, float eps) {
  using P = Pack<DT>;
  constexpr int E = P::E;
  __shared__ Stats s_warp[32];

  const int rows_per_cta = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const long long row = static_cast<long long>(blockIdx.x) * rows_per_cta + slot;
  const bool row_ok = row < rows;
  const long long base = row * nvec;

  // Issue every load of this thread's slice of the row before using any.
  uint4 xv[VPT], rv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = t + i * tpr;
    xv[i] = make_uint4(0, 0, 0, 0);
    rv[i] = make_uint4(0, 0, 0, 0);
    if (row_ok && c < nvec) {
      xv[i] = ld_stream(x + base + c);
      if (r) rv[i] = ld_stream(r + base + c);
    }
  }

  // Levels 1-2, incremental: fold each 16-byte block into the running stats.
  float h[VPT][E];
  Stats st{0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    float xf[E], rf_[E];
    P::unpack(xv[i], xf);
    P::unpack(rv[i], rf_);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      h[i][e] = xf[e] + rf_[e];
      s += h[i][e];
    }
    const float mb = s * (1.0f / E);
    float q = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float d = h[i][e] - mb;
      q = fmaf(d, d, q);
    }
    if (t + i * tpr < nvec) st = chan(st, Stats{float(E), mb, q});
  }
  // Merge the threads of the warp (all 32 lanes belong to this row).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stats b{__shfl_xor_sync(0xffffffffu, st.n, o), __shfl_xor_sync(0xffffffffu, st.mean, o),
            __shfl_xor_sync(0xffffffffu, st.m2, o)};
    st = chan(st, b);
  }
  // Merge the warps of the row through shared memory (same order in every thread).
  const int warps_per_row = tpr >> 5;
  if (warps_per_row > 1) {
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) s_warp[w] = st;
    __syncthreads();
    const int w0 = slot * warps_per_row;
    st = s_warp[w0];
    for (int j = 1; j < warps_per_row; ++j) st = chan(st, s_warp[w0 + j]);
  }
  if (!row_ok) return;

  // Level 3: normalise and apply the affine map from registers.
  const float mean = st.mean;
  const float rstd = rsqrtf(st.m2 * inv_cols + eps);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = t + i * tpr;
    if (c >= nvec) continue;
    float g[E], b[E], y[E];
    if (gamma) {
      P::unpack(__ldg(gamma + c), g);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = 1.f;
    }
    if (beta) {
      P::unpack(__ldg(beta + c), b);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) b[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = fmaf((h[i][e] - mean) * rstd, g[e], b[e]);
    st_stream(out + base + c, P::pack(y));
    if (r_out) st_stream(r_out + base + c, P::pack(h[i]));
  }
}

template <Dt DT>
cudaError_t launch_dt(const void* x, const void* r, const void* g, const void* b, void* out, void* r_out,
                      int rows, int cols, float eps, cudaStream_t s) {
  constexpr int E = Pack<DT>::E;
  const int nvec = cols / E;
  const int vpt = nvec >= 256 ? 4 : (nvec >= 64 ? 2 : 1);
  int tpr = (nvec + vpt - 1) / vpt;
  tpr = (tpr + 31) & ~31;
  const int rows_per_cta = tpr >= 256 ? 1 : 256 / tpr;
  const int threads = tpr * rows_per_cta;
  const long long grid = (static_cast<long long>(rows) + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const float inv_cols = 1.0f / static_cast<float>(cols);
  auto X = static_cast<const uint4*>(x);
  auto R = static_cast<const uint4*>(r);
  auto G = static_cast<const uint4*>(g);
  auto Bt = static_cast<const uint4*>(b);
  auto O = static_cast<uint4*>(out);
  auto RO = static_cast<uint4*>(r_out);
  if (vpt == 4)
    ln_fused_kernel<DT, 4><<<unsigned(grid), threads, 0, s>>>(X, R, G, Bt, O, RO, rows, nvec, tpr, inv_cols, eps);
  else if (vpt == 2)
    ln_fused_kernel<DT, 2><<<unsigned(grid), threads, 0, s>>>(X, R, G, Bt, O, RO, rows, nvec, tpr, inv_cols, eps);
  else
    ln_fused_kernel<DT, 1><<<unsigned(grid), threads, 0, s>>>(X, R, G, Bt, O, RO, rows, nvec, tpr, inv_cols, eps);
  return cudaGetLastError();
}

}  // namespace

// 1024 threads x 4 vectors of 16 bytes per row at most.
int layernorm_max_cols(Dt dt) { return 1024 * 4 * (dt == Dt::F32 ? 4 : 8); }

cudaError_t launch_layernorm(const void* x, const void* r, const void* gamma, const void* beta, void* out,
                             void* r_out, int rows, int cols, float eps, Dt dt, cudaStream_t s) {
  switch (dt) {
    case Dt::F32: return launch_dt<Dt::F32>(x, r, gamma, beta, out, r_out, rows, cols, eps, s);
    case Dt::F16: return launch_dt<Dt::F16>(x, r, gamma, beta, out, r_out, rows, cols, eps, s);
    case Dt::BF16: return launch_dt<Dt::BF16>(x, r, gamma, beta, out, r_out, rows, cols, eps, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rf
