// ln_fused.cu -- one-pass residual + LayerNorm and residual + RMSNorm
// ("Operator Fusion" guide,
// section 1 traffic example and section 2 Pattern 2: mean -> variance ->
// normalise; section 4 places eps inside the square root).
//
// The cascade mean -> M2 -> normalise runs fused in one pass, in the
// incremental form of RedFuser (Figure 4): level 2's dependence on level 1 is
// the additive correction M2 = sum((h - K)^2) - n (mean - K)^2 for any shift
// K, so with one shift K for the whole row both levels are plain running sums,
// S1 = sum(h - K) and S2 = sum((h - K)^2), updated as each element arrives and
// merged across lanes (shuffles) and warps (shared memory) with combine op +;
// then mean - K = S1/n and M2 = S2 - S1^2/n once per row.  (A per-thread
// shift would need Chan, Golub and LeVeque's pairwise combine of
// (n, mean, M2) at every merge step; a common shift turns it into two sums,
// and the per-row merge was this kernel's serial latency.)
//
// Accuracy.  S2 carries rounding of the order of u * S2 = u * (M2 + n d^2),
// d = mean - K, so the subtraction loses about log2(1 + n d^2 / M2) bits.  K
// is the mean of the row's first 16-byte vector, which every thread of the row
// reads: for a row of exchangeable values n d^2 / M2 is then of the order of
// 1/8 (bf16/f16) or 1/4 (fp32).  When a row still has n d^2 > M2 (an outlier
// among its first elements), the row takes a second reduction over the values
// already in registers, M2 = sum((h - K - d)^2), which does not cancel.  With
// n d^2 <= M2 the one-pass M2 is within a few dozen ulps, and the
// normalisation uses (h - K) - d, which keeps the large-mean case exact where
// h - mean, with mean rounded to fp32, would not.  The row stays in registers
// between the statistics and the normalisation, so x and the residual are read
// from HBM once and y is written once.
//
// The kernel is bound by instruction issue as much as by HBM, so the
// element-wise work runs on packed fp32 pairs (fma/add/mul .f32x2): three
// packed operations per pair for the statistics.  The affine map keeps the
// centred form y = ((h - K) - (mean - K)) * (gamma * rstd) + beta; a row of
// equal values gets K equal to that value, hence exactly beta.
//
// Layout: a group of `tpr` threads (a multiple of 32) owns one row; thread t
// holds the row's 16-byte vectors t, t + tpr, ..., t + (VPT-1)*tpr.  A CTA
// holds max(1, 256 / tpr) rows.
#include "rf_device.cuh"

namespace rf {
namespace {

// 16-byte vector <-> packed fp32 pairs.
template <Dt DT>
struct Vec2;

template <>
struct Vec2<Dt::BF16> {
  static constexpr int P = 4;  // pairs per 16 bytes
  __device__ __forceinline__ static void unpack(const uint4& u, uint64_t* p) {
    p[0] = u2pack(u.x << 16, u.x & 0xffff0000u);
    p[1] = u2pack(u.y << 16, u.y & 0xffff0000u);
    p[2] = u2pack(u.z << 16, u.z & 0xffff0000u);
    p[3] = u2pack(u.w << 16, u.w & 0xffff0000u);
  }
  __device__ __forceinline__ static uint32_t pack1(uint64_t v) {
    float lo, hi;
    f2unpack(v, lo, hi);
    return pack_bf16x2(lo, hi);
  }
  __device__ __forceinline__ static uint4 pack(const uint64_t* p) {
    return make_uint4(pack1(p[0]), pack1(p[1]), pack1(p[2]), pack1(p[3]));
  }
};

template <>
struct Vec2<Dt::F16> {
  static constexpr int P = 4;
  __device__ __forceinline__ static uint64_t up1(uint32_t w) {
    const float2 f = unpack_f16x2(w);
    return f2pack(f.x, f.y);
  }
  __device__ __forceinline__ static void unpack(const uint4& u, uint64_t* p) {
    p[0] = up1(u.x);
    p[1] = up1(u.y);
    p[2] = up1(u.z);
    p[3] = up1(u.w);
  }
  __device__ __forceinline__ static uint32_t pack1(uint64_t v) {
    float lo, hi;
    f2unpack(v, lo, hi);
    return pack_f16x2(lo, hi);
  }
  __device__ __forceinline__ static uint4 pack(const uint64_t* p) {
    return make_uint4(pack1(p[0]), pack1(p[1]), pack1(p[2]), pack1(p[3]));
  }
};

template <>
struct Vec2<Dt::F32> {
  static constexpr int P = 2;
  __device__ __forceinline__ static void unpack(const uint4& u, uint64_t* p) {
    p[0] = u2pack(u.x, u.y);
    p[1] = u2pack(u.z, u.w);
  }
  __device__ __forceinline__ static uint4 pack(const uint64_t* p) {
    uint4 u;
    f2unpack_u(p[0], u.x, u.y);
    f2unpack_u(p[1], u.z, u.w);
    return u;
  }
};

__device__ __forceinline__ float hsum(uint64_t v) {
  float lo, hi;
  f2unpack(v, lo, hi);
  return lo + hi;
}

// Named barrier over the `count` threads of one row (ids 1..; 0 is __syncthreads).
__device__ __forceinline__ void row_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// R_OUT: h = x + r is also written out; otherwise the registers keep h - K,
// which the normalisation uses directly.
template <Dt DT, int VPT, bool R_OUT>
__global__ void __launch_bounds__(1024) ln_fused_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                        const uint4* __restrict__ gamma,
                                                        const uint4* __restrict__ beta, uint4* __restrict__ out,
                                                        uint4* __restrict__ r_out, int rows, int nvec, int tpr,
                                                        float inv_cols, float eps, unsigned* status) {
  using V = Vec2<DT>;
  constexpr int P = V::P;
  __shared__ float2 s_warp[32];

  const int rows_per_cta = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const long long row = static_cast<long long>(blockIdx.x) * rows_per_cta + slot;
  // the row's vectors t, t + tpr, ... must cover [0, nvec) within the tensor
  const bool row_ok = row < rows && RF_INB(t < tpr && VPT * tpr >= nvec && slot < rows_per_cta, status);
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

  // Levels 1-2, incremental: running sums about K, the mean of the row's first
  // 16-byte vector (valid blocks form a prefix i < count; blocks past the row
  // end are skipped).
  float shift = 0.f;
  if (row_ok) {
    uint64_t x0[P], r0[P];
    V::unpack(__ldg(x + base), x0);
    if (r) {
      V::unpack(__ldg(r + base), r0);
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) r0[k] = 0;
    }
    // a pairwise tree, so that a row of equal values gets exactly that value
    uint64_t hp[P];
#pragma unroll
    for (int k = 0; k < P; ++k) hp[k] = add_f32x2(x0[k], r0[k]);
#pragma unroll
    for (int w = P / 2; w > 0; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) hp[k] = add_f32x2(hp[k], hp[k + w]);
    shift = hsum(hp[0]) * (1.0f / (2 * P));
  }
  const uint64_t negk2 = f2pack(-shift, -shift);
  uint64_t h[VPT][P];
  uint64_t s1 = 0, s2 = 0;  // packed pairs: two partial sums each
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    uint64_t xp[P], rp[P];
    V::unpack(xv[i], xp);
    V::unpack(rv[i], rp);
    const bool valid = t + i * tpr < nvec;
#pragma unroll
    for (int k = 0; k < P; ++k) {
      const uint64_t hv = add_f32x2(xp[k], rp[k]);
      const uint64_t d = add_f32x2(hv, negk2);
      h[i][k] = R_OUT ? hv : d;
      if (valid) {
        s1 = add_f32x2(s1, d);
        s2 = fma_f32x2(d, d, s2);
      }
    }
  }
  float a1 = hsum(s1), a2 = hsum(s2);
  // Merge the threads of the warp (all 32 lanes belong to this row): combine op +.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
  }
  // Merge the warps of the row through shared memory (same order in every thread).
  const int warps_per_row = tpr >> 5;
  if (warps_per_row > 1) {
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) s_warp[w] = make_float2(a1, a2);
    __syncthreads();
    const int w0 = slot * warps_per_row;
    float2 acc = s_warp[w0];
    for (int j = 1; j < warps_per_row; ++j) {
      acc.x += s_warp[w0 + j].x;
      acc.y += s_warp[w0 + j].y;
    }
    a1 = acc.x;
    a2 = acc.y;
  }
  const float mean_k = a1 * inv_cols;  // mean - K
  float var = fmaxf(fmaf(-mean_k, mean_k, a2 * inv_cols), 0.f);
  const uint64_t negmk2 = f2pack(-mean_k, -mean_k);
  // Rows whose shift lies more than one standard deviation from their mean
  // recompute M2 about the mean from registers.  Every thread of a row holds
  // the same sums, so the decision is uniform over the row; the row's warps
  // merge through a named barrier of their own, and other rows do not wait.
  if (mean_k * mean_k > var) {
    uint64_t q2 = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (t + i * tpr >= nvec) continue;
#pragma unroll
      for (int k = 0; k < P; ++k) {
        const uint64_t e = add_f32x2(R_OUT ? add_f32x2(h[i][k], negk2) : h[i][k], negmk2);
        q2 = fma_f32x2(e, e, q2);
      }
    }
    float m2 = hsum(q2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
    if (warps_per_row > 1) {
      const int w = threadIdx.x >> 5;
      row_barrier(1 + slot, tpr);  // the row's threads have read the first merge's values
      if ((threadIdx.x & 31) == 0) s_warp[w].x = m2;
      row_barrier(1 + slot, tpr);
      const int w0 = slot * warps_per_row;
      m2 = s_warp[w0].x;
      for (int j = 1; j < warps_per_row; ++j) m2 += s_warp[w0 + j].x;
    }
    var = m2 * inv_cols;
  }
  if (!row_ok) return;

  // Level 3: y = ((h - K) - (mean - K)) * (gamma * rstd) + beta: three packed
  // ops per pair from h - K (four when h itself is kept for residual_out).
  const float rstd = rsqrtf(var + eps);
  const uint64_t rstd2 = f2pack(rstd, rstd);
  const uint64_t one2 = f2pack(1.f, 1.f), zero2 = 0;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = t + i * tpr;
    if (c >= nvec) continue;
    uint64_t g[P], b[P], y[P];
    if (gamma) {
      V::unpack(__ldg(gamma + c), g);
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) g[k] = one2;
    }
    if (beta) {
      V::unpack(__ldg(beta + c), b);
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) b[k] = zero2;
    }
#pragma unroll
    for (int k = 0; k < P; ++k) {
      const uint64_t a = mul_f32x2(g[k], rstd2);
      y[k] = fma_f32x2(add_f32x2(R_OUT ? add_f32x2(h[i][k], negk2) : h[i][k], negmk2), a, b[k]);
    }
    st_stream(out + base + c, V::pack(y));
    if (R_OUT) st_stream(r_out + base + c, V::pack(h[i]));
  }
}


// RMSNorm: the one-level cascade sum(h^2) -> normalise.  Each thread folds its
// 16-byte blocks into a running sum of squares (combine op +), the threads of
// a row are summed by warp shuffles and then across warps in shared memory,
// and y = h * (gamma * rsqrt(sum / n + eps)) is written from registers.
template <Dt DT, int VPT>
__global__ void __launch_bounds__(1024) rms_fused_kernel(const uint4* __restrict__ x, const uint4* __restrict__ r,
                                                         const uint4* __restrict__ gamma, uint4* __restrict__ out,
                                                         uint4* __restrict__ r_out, int rows, int nvec, int tpr,
                                                         float inv_cols, float eps, unsigned* status) {
  using V = Vec2<DT>;
  constexpr int P = V::P;
  __shared__ float s_warp[32];

  const int rows_per_cta = blockDim.x / tpr;
  const int slot = threadIdx.x / tpr;
  const int t = threadIdx.x - slot * tpr;
  const long long row = static_cast<long long>(blockIdx.x) * rows_per_cta + slot;
  // the row's vectors t, t + tpr, ... must cover [0, nvec) within the tensor
  const bool row_ok = row < rows && RF_INB(t < tpr && VPT * tpr >= nvec && slot < rows_per_cta, status);
  const long long base = row * nvec;

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
  uint64_t h[VPT][P];
  uint64_t q2 = 0;  // running sum of squares, two lanes of a packed pair
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    uint64_t xp[P], rp[P];
    V::unpack(xv[i], xp);
    V::unpack(rv[i], rp);
#pragma unroll
    for (int k = 0; k < P; ++k) {
      h[i][k] = add_f32x2(xp[k], rp[k]);
      q2 = fma_f32x2(h[i][k], h[i][k], q2);  // blocks past the row end are zero
    }
  }
  float ss = hsum(q2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const int warps_per_row = tpr >> 5;
  if (warps_per_row > 1) {
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) s_warp[w] = ss;
    __syncthreads();
    const int w0 = slot * warps_per_row;
    ss = s_warp[w0];
    for (int j = 1; j < warps_per_row; ++j) ss += s_warp[w0 + j];
  }
  if (!row_ok) return;
  const float rstd = rsqrtf(ss * inv_cols + eps);
  const uint64_t rstd2 = f2pack(rstd, rstd);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = t + i * tpr;
    if (c >= nvec) continue;
    uint64_t g[P], y[P];
    if (gamma) {
      V::unpack(__ldg(gamma + c), g);
    } else {
#pragma unroll
      for (int k = 0; k < P; ++k) g[k] = f2pack(1.f, 1.f);
    }
#pragma unroll
    for (int k = 0; k < P; ++k) y[k] = mul_f32x2(h[i][k], mul_f32x2(g[k], rstd2));
    st_stream(out + base + c, V::pack(y));
    if (r_out) st_stream(r_out + base + c, V::pack(h[i]));
  }
}

template <Dt DT, bool RMS>
cudaError_t launch_dt(const void* x, const void* r, const void* g, const void* b, void* out, void* r_out,
                      int rows, int cols, float eps, unsigned* status, cudaStream_t s) {
  constexpr int E = 2 * Vec2<DT>::P;
  const int nvec = cols / E;
  const int vpt = nvec >= 128 ? 4 : (nvec >= 64 ? 2 : 1);  // one warp per row from 128 vectors up
  int tpr = (nvec + vpt - 1) / vpt;
  tpr = (tpr + 31) & ~31;
  // rows per CTA (4096 bf16 columns, 128 threads per row): LayerNorm 2 (65.1 us;
  // 1: 80.7, 4: 69.0), RMSNorm 1 (58.1 us; 2: 59.4, 4: 61.4)
  const int rows_per_cta = tpr >= 256 ? 1 : (RMS ? max(1, 128 / tpr) : 256 / tpr);
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
  const unsigned gr = static_cast<unsigned>(grid);
  if constexpr (RMS) {
    if (vpt == 4)
      rms_fused_kernel<DT, 4><<<gr, threads, 0, s>>>(X, R, G, O, RO, rows, nvec, tpr, inv_cols, eps, status);
    else if (vpt == 2)
      rms_fused_kernel<DT, 2><<<gr, threads, 0, s>>>(X, R, G, O, RO, rows, nvec, tpr, inv_cols, eps, status);
    else
      rms_fused_kernel<DT, 1><<<gr, threads, 0, s>>>(X, R, G, O, RO, rows, nvec, tpr, inv_cols, eps, status);
  } else {
#define RF_LN(V_, RO_) ln_fused_kernel<DT, V_, RO_><<<gr, threads, 0, s>>>(X, R, G, Bt, O, RO, rows, nvec, tpr, inv_cols, eps, status)
    if (RO) {
      if (vpt == 4) RF_LN(4, true); else if (vpt == 2) RF_LN(2, true); else RF_LN(1, true);
    } else {
      if (vpt == 4) RF_LN(4, false); else if (vpt == 2) RF_LN(2, false); else RF_LN(1, false);
    }
#undef RF_LN
  }
  return cudaGetLastError();
}

}  // namespace

// 1024 threads x 4 vectors of 16 bytes per row at most.
int layernorm_max_cols(Dt dt) { return 1024 * 4 * (dt == Dt::F32 ? 4 : 8); }

cudaError_t launch_layernorm(const void* x, const void* r, const void* gamma, const void* beta, void* out,
                             void* r_out, int rows, int cols, float eps, Dt dt, unsigned* status, cudaStream_t s) {
  switch (dt) {
    case Dt::F32: return launch_dt<Dt::F32, false>(x, r, gamma, beta, out, r_out, rows, cols, eps, status, s);
    case Dt::F16: return launch_dt<Dt::F16, false>(x, r, gamma, beta, out, r_out, rows, cols, eps, status, s);
    case Dt::BF16: return launch_dt<Dt::BF16, false>(x, r, gamma, beta, out, r_out, rows, cols, eps, status, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_rmsnorm(const void* x, const void* r, const void* gamma, void* out, void* r_out, int rows, int cols,
                           float eps, Dt dt, unsigned* status, cudaStream_t s) {
  switch (dt) {
    case Dt::F32: return launch_dt<Dt::F32, true>(x, r, gamma, nullptr, out, r_out, rows, cols, eps, status, s);
    case Dt::F16: return launch_dt<Dt::F16, true>(x, r, gamma, nullptr, out, r_out, rows, cols, eps, status, s);
    case Dt::BF16: return launch_dt<Dt::BF16, true>(x, r, gamma, nullptr, out, r_out, rows, cols, eps, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rf
