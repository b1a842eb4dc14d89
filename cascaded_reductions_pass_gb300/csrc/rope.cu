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
// Angles: see rope_angle.cuh (accurate p * base^(-2i/D), reduced modulo
// 2 pi, then the hardware sine and cosine on the reduced angle).  Each CTA builds a cos/sin table for its positions in
// shared memory and reuses it across all (batch, head) rows.
//
// Work: a thread takes one pair of 16-byte chunks of a row (dims c*8..c*8+7
// and the same dims + D/2), four pairs at a time so that eight loads are in
// flight.  In place is allowed: each thread writes exactly what it read.
#include "rf_device.cuh"
#include "rope_angle.cuh"

namespace rf {

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
  for (int e = 0; e < 8; ++e) rope_rotate(xa[e], xb[e], cs[e * stride], ya[e], yb[e]);
  b_out = Pack<DT>::pack(yb);
  return Pack<DT>::pack(ya);
}

// The rows of one CTA: (tensor, batch*head, position) x chunk pair, as a 32-bit
// index; NBC is the CTA's position count when known at compile time (every
// block but the last), so the index splits without a runtime division there.
template <Dt DT, int D, int NBC>
__device__ __forceinline__ void rotate_rows(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                            uint4* __restrict__ qo, uint4* __restrict__ ko, int BHq, int BHkv,
                                            int N, int n0, int nb_rt, const float2* cs, unsigned* status) {
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
      if (live[u]) live[u] = RF_INB(bh < (isq[u] ? BHq : BHkv) && n0 + nl[u] < N && nl[u] < nb, status);
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
                                                        const __grid_constant__ RopeParams prm, unsigned* status) {
  constexpr int H2 = D / 2;
  constexpr int CP = CsLayout<D>::CP, RS = CsLayout<D>::RS;
  __shared__ float2 cs[kNB * RS];
  const int n0 = blockIdx.x * kNB;
  const int nb = min(kNB, N - n0);
  for (int e = threadIdx.x; e < kNB * H2; e += kThreads) {
    const int nl = e / H2, i = e - nl * H2;
    cs[nl * RS + (i & 7) * CP + (i >> 3)] = rope_cs(static_cast<float>(pos_offset + n0 + nl), i, prm);
  }
  __syncthreads();

  if (nb == kNB) {
    rotate_rows<DT, D, kNB>(q, k, qo, ko, BHq, BHkv, N, n0, kNB, cs, status);
  } else {
    rotate_rows<DT, D, 0>(q, k, qo, ko, BHq, BHkv, N, n0, nb, cs, status);
  }
}

template <Dt DT>
cudaError_t launch_dt(const void* q, const void* k, void* qo, void* ko, int BHq, int BHkv, int N, int D,
                      int pos_offset, const RopeParams& prm, unsigned* status, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((N + kNB - 1) / kNB);
  auto Q = static_cast<const uint4*>(q);
  auto K = static_cast<const uint4*>(k);
  auto QO = static_cast<uint4*>(qo);
  auto KO = static_cast<uint4*>(ko);
  switch (D) {
    case 64: rope_kernel<DT, 64><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm, status); break;
    case 128: rope_kernel<DT, 128><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm, status); break;
    case 256: rope_kernel<DT, 256><<<grid, kThreads, 0, s>>>(Q, K, QO, KO, BHq, BHkv, N, pos_offset, prm, status); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_qk(const void* q, const void* k, void* q_out, void* k_out, int BHq, int BHkv, int N, int D,
                           double base, int pos_offset, Dt dt, unsigned* status, cudaStream_t s) {
  const RopeParams prm = make_rope_params(base, D);
  switch (dt) {
    case Dt::F16: return launch_dt<Dt::F16>(q, k, q_out, k_out, BHq, BHkv, N, D, pos_offset, prm, status, s);
    case Dt::BF16: return launch_dt<Dt::BF16>(q, k, q_out, k_out, BHq, BHkv, N, D, pos_offset, prm, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rf
