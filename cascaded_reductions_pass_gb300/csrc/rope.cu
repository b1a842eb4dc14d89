// rope.cu -- rotary position embedding of Q and K (the pre-matmul
// transformation of AttnFuse, Abstract and Figure 1), as one HBM pass before
// the attention kernel.
//
// For head dimension D and i < D/2 the pair (x_i, x_{i+D/2}) of a row at
// position p turns by theta = p * base^(-2i/D) (the rotate-half pairing).
//
// Why a separate pass on this GPU: AttnFuse's "Rotation Calculus" (Table 4)
// finds that whether fusing RoPE into the attention kernel pays depends on the
// compute-to-bandwidth ratio.  In the tcgen05 attention kernel K reaches the
// tensor core straight from TMA-written shared memory, so a fused rotation of
// K would be redone by every CTA that streams the tile (N / 256 times), on the
// issue slots that already bound the D = 64 kernel; one pass over Q and K
// costs their bytes twice at HBM speed instead.
//
// Angles: the host passes base^(-2i/D) computed in double and split into two
// floats (hi + lo).  The kernel forms p * (hi + lo) as a float pair (the
// product's rounding error recovered with an FMA), reduces it modulo 2 pi by
// Cody and Waite's method with 2 pi split into three floats, and calls
// sincosf on the reduced angle, so positions in the tens of thousands keep
// angle errors near 1e-7.  Each CTA builds a cos/sin table for its positions
// in shared memory and reuses it across all (batch, head) rows.
//
// Work: a thread takes one pair of 16-byte chunks of a row (dims c*8..c*8+7
// and the same dims + D/2), four pairs at a time so that eight loads are in
// flight.  In place is allowed: each thread writes exactly what it read.
#include "rf_device.cuh"

namespace rf {

struct RopeParams {
  float fhi[kRopeMaxHalf], flo[kRopeMaxHalf];  // base^(-2i/D) = fhi[i] + flo[i]
  float two_pi[3];                             // 2 pi = sum of the three floats
  float inv_two_pi;
};

namespace {

constexpr int kNB = 2;         // positions per CTA (small CTAs: many in flight, no long tail)
constexpr int kThreads = 128;
constexpr int kUnroll = 4;

// Shared cos/sin table of a CTA, laid out [position][e][chunk pair] (angle
// index i = chunk pair * 8 + e) with a 32-byte pad per position: a warp's 32
// items (consecutive chunk pairs of consecutive positions) then read 32
// distinct 8-byte slots in the minimum two shared-memory wavefronts for
// D = 64, 128 and 256 ([position][i] put every position at the same banks).
template <int D>
struct CsLayout {
  static constexpr int CP = D / 16;
  static constexpr int RS = 8 * CP + 4;  // float2 per position row, padded
};

template <Dt DT>
__device__ __forceinline__ uint4 rotate(const uint4& a, const uint4& b, const float2* cs, int stride, uint4& b_out) {
  float xa[8], xb[8], ya[8], yb[8];
  Pack<DT>::unpack(a, xa);
  Pack<DT>::unpack(b, xb);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 t = cs[e * stride];  // (cos, sin)
    ya[e] = fmaf(xa[e], t.x, -xb[e] * t.y);
    yb[e] = fmaf(xa[e], t.y, xb[e] * t.x);
  }
  b_out = Pack<DT>::pack(yb);
  return Pack<DT>::pack(ya);
}

// The rows of one CTA: (tensor, batch*head, position) x chunk pair, as a 32-bit
// index; NBC is the CTA's position count when known at compile time (every
// block but the last), so the index splits without a runtime division there.
template <Dt DT, int D, int NBC>
__device__ __forceinline__ void rotate_rows(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                            uint4* __restrict__ qo, uint4* __restrict__ ko, int BHq, int BHkv,
                                            int N, int n0, int nb_rt, const float2* cs) {
  constexpr int CP = D / 16;  // chunk pairs per row
  constexpr int RS = CsLayout<D>::RS;
  constexpr int RV = D / 8;   // 16-byte chunks per row
  const int nb = NBC ? NBC : nb_rt;
  const int per_q = BHq * nb * CP;
  const int items = per_q + (k ? BHkv * nb * CP : 0);
  for (int it0 = threadIdx.x; it0 < items; it0 += kThreads * kUnroll) {
    uint4 a[kUnroll], b[kUnroll];
    long long row[kUnroll];
    int cp[kUnroll], nl[kUnroll];
    bool isq[kUnroll], live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int it = it0 + u * kThreads;
      live[u] = it < items;
      isq[u] = it < per_q;
      const int j = (isq[u] ? it : it - per_q);
      cp[u] = j % CP;
      const int r = j / CP;
      const int bh = r / nb;
      nl[u] = r - bh * nb;
      row[u] = (static_cast<long long>(bh) * N + n0 + nl[u]) * RV;
      if (live[u]) {
        const uint4* src = isq[u] ? q : k;
        a[u] = ld_stream(src + row[u] + cp[u]);
        b[u] = ld_stream(src + row[u] + cp[u] + CP);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (!live[u]) continue;
      uint4 yb;
      const uint4 ya = rotate<DT>(a[u], b[u], cs + nl[u] * RS + cp[u], CP, yb);
      uint4* dst = isq[u] ? qo : ko;
      st_stream(dst + row[u] + cp[u], ya);
      st_stream(dst + row[u] + cp[u] + CP, yb);
    }
  }
}

template <Dt DT, int D>
__global__ void __launch_bounds__(kThreads) rope_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                                        uint4* __restrict__ qo, uint4* __restrict__ ko, int BHq,
                                                        int BHkv, int N, int pos_offset,
                                                        const __grid_constant__ RopeParams prm) {
  constexpr int H2 = D / 2;
  constexpr int CP = CsLayout<D>::CP, RS = CsLayout<D>::RS;
  __shared__ float2 cs[kNB * RS];
  const int n0 = blockIdx.x * kNB;
  const int nb = min(kNB, N - n0);
  for (int e = threadIdx.x; e < kNB * H2; e += kThreads) {
    const int nl = e / H2, i = e - nl * H2;
    // theta = p * (fhi + flo) as th + tl, then th + tl - j * 2 pi with j = nearest integer
    const float p = static_cast<float>(pos_offset + n0 + nl);
    const float th = p * prm.fhi[i];
    const float tl = fmaf(p, prm.flo[i], fmaf(p, prm.fhi[i], -th));
    const float j = rintf(th * prm.inv_two_pi);
    float r = fmaf(-j, prm.two_pi[0], th);
    r = fmaf(-j, prm.two_pi[1], r);
    r = fmaf(-j, prm.two_pi[2], r);
    r += tl;
    float s, c;
    sincosf(r, &s, &c);
    cs[nl * RS + (i & 7) * CP + (i >> 3)] = make_float2(c, s);
  }
  __syncthreads();

  if (nb == kNB) {
    rotate_rows<DT, D, kNB>(q, k, qo, ko, BHq, BHkv, N, n0, kNB, cs);
  } else {
    rotate_rows<DT, D, 0>(q, k, qo, ko, BHq, BHkv, N, n0, nb, cs);
  }
}

template <Dt DT>
cudaError_t launch_dt(const void* q, const void* k, void* qo, void* ko, int BHq, int BHkv, int N, int D,
                      int pos_offset, const RopeParams& prm, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((N + kNB - 1) / kNB);
  auto Q = static_cast<const uint4*>(q);
  auto K = static_cast<const uint4*>(k);
  auto QO = static_cast<uint4*>(qo);
  auto KO = static_cast<uint4*>(ko);
  switch (D) {
    case 64: rope_kernel<DT, 64><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm); break;
    case 128: rope_kernel<DT, 128><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm); break;
    case 256: rope_kernel<DT, 256><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_qk(const void* q, const void* k, void* q_out, void* k_out, int BHq, int BHkv, int N, int D,
                           double base, int pos_offset, Dt dt, cudaStream_t s) {
  RopeParams prm;
  const int half = D / 2;
  for (int i = 0; i < kRopeMaxHalf; ++i) {
    const double f = i < half ? pow(base, -2.0 * i / D) : 0.0;
    prm.fhi[i] = static_cast<float>(f);
    prm.flo[i] = static_cast<float>(f - static_cast<double>(prm.fhi[i]));
  }
  const double two_pi = 2.0 * 3.14159265358979323846;
  prm.two_pi[0] = static_cast<float>(two_pi);
  prm.two_pi[1] = static_cast<float>(two_pi - static_cast<double>(prm.two_pi[0]));
  prm.two_pi[2] = static_cast<float>(two_pi - static_cast<double>(prm.two_pi[0]) - static_cast<double>(prm.two_pi[1]));
  prm.inv_two_pi = static_cast<float>(1.0 / two_pi);
  switch (dt) {
    case Dt::F16: return launch_dt<Dt::F16>(q, k, q_out, k_out, BHq, BHkv, N, D, pos_offset, prm, s);
    case Dt::BF16: return launch_dt<Dt::BF16>(q, k, q_out, k_out, BHq, BHkv, N, D, pos_offset, prm, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rf
