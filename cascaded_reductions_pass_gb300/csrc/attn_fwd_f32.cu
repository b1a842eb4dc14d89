// attn_fwd_f32.cu -- exact fp32 attention forward on the FP32 pipes (SIMT).
//
// The cascade max -> sum exp -> sum exp * v (RedFuser, Abstract: safe softmax
// followed by GEMM) fused into one loop over key tiles in the incremental
// form (RedFuser, Figure 4): for each tile of 32 keys the running row max m
// (level 1, reduce max / combine +) is raised, the running sum l and the
// running output acc (levels 2-3, reduce + / combine *) are rescaled by
// exp(m_old - m_new) and the tile's terms are added.  O = acc / l and
// LSE = m + ln l at the end.  fp32 tensor-core modes (TF32) round the
// operands to 10 mantissa bits, too coarse for a 1e-5 relative result, so
// this path uses FFMA throughout with the accurate expf/logf.
//
// CTA: 4 warps, 16 query rows (4 per warp), key tiles of 32 (one key per
// lane) staged in shared memory with K rows padded to D+4 floats.  Each warp
// forms the scores of its four rows together, so a lane reads its key's K row
// once per tile for all four; the exponentials are base 2 (log2 e folded into
// the scale) through exp2f, accurate to 2 ulp; the probabilities go through
// shared memory, where the output update reads four keys of a row with one
// broadcast load.  With the causal mask a sliding window (key j visible to
// query i iff i - window < j) and ALiBi biases (+ slope_h * (j - i)) are
// supported as in the tensor-core path.
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 4;
constexpr int kBM = kRowsPerWarp * kWarps;  // 16 query rows per CTA
constexpr int kBN = 32;                     // keys per tile

template <int DC>  // DC = ceil(D / 32) output columns per lane
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const float* __restrict__ q,
                                                               const float* __restrict__ k,
                                                               const float* __restrict__ v, float* __restrict__ o,
                                                               float* __restrict__ lse, int Hq, int Hkv, int Nq,
                                                               int Nk, int D, float scale, int causal, int window,
                                                               const float* __restrict__ alibi, unsigned* status) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  const int KS = D + 4;               // padded K row stride (floats)
  float* Qs = smem;                   // [kBM][D]
  float* Ks = Qs + kBM * D;           // [kBN][KS]
  float* Vs = Ks + kBN * KS;          // [kBN][D]
  float* Ps = Vs + kBN * D;           // [kWarps][kRowsPerWarp][kBN] probabilities of the tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y, hk = h / (Hq / Hkv);
  const int q0 = blockIdx.x * kBM;
  // the grid is (query blocks, Hq, B): a block past them has nothing to do
  if (!RF_INB(q0 < Nq && h < Hq && hk < Hkv && D <= 32 * DC, status)) return;
  const float* qh = q + (static_cast<long long>(b) * Hq + h) * Nq * D;
  const float* kh = k + (static_cast<long long>(b) * Hkv + hk) * Nk * D;
  const float* vh = v + (static_cast<long long>(b) * Hkv + hk) * Nk * D;
  const int D4 = D >> 2;
  constexpr float kLog2e = 1.4426950408889634f;
  const float sl2 = scale * kLog2e;  // scores in base-2 units

  for (int i = threadIdx.x; i < kBM * D4; i += blockDim.x) {
    const int r = i / D4, c = i - r * D4;
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + r < Nq) val = reinterpret_cast<const float4*>(qh + static_cast<long long>(q0 + r) * D)[c];
    reinterpret_cast<float4*>(Qs + r * D)[c] = val;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DC];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) acc[r][c] = 0.f;
  }

  const int last_row = min(q0 + kBM, Nq) - 1;
  const int kend = causal ? min(Nk, last_row + 1) : Nk;  // keys past the CTA's last row are all masked
  // a sliding window hides every key below the first row's window
  const int kbeg = (causal && window > 0) ? (max(0, q0 - window + 1) / kBN) * kBN : 0;
  const float slope2 = alibi ? __ldg(alibi + h) * kLog2e : 0.f;
  const float* qw_rows = Qs + warp * kRowsPerWarp * D;
  float* pw = Ps + warp * kRowsPerWarp * kBN;
  for (int k0 = kbeg; k0 < kend; k0 += kBN) {
    __syncthreads();
    for (int i = threadIdx.x; i < kBN * D4; i += blockDim.x) {
      const int r = i / D4, c = i - r * D4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (k0 + r < Nk) {
        kv = reinterpret_cast<const float4*>(kh + static_cast<long long>(k0 + r) * D)[c];
        vv = reinterpret_cast<const float4*>(vh + static_cast<long long>(k0 + r) * D)[c];
      }
      reinterpret_cast<float4*>(Ks + r * KS)[c] = kv;
      reinterpret_cast<float4*>(Vs + r * D)[c] = vv;
    }
    __syncthreads();

    // scores of the warp's four rows against this lane's key
    const int key = k0 + lane;
    float dot[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) dot[r] = 0.f;
    const float* kr = Ks + lane * KS;
    for (int d = 0; d < D; d += 4) {
      const float4 c = *reinterpret_cast<const float4*>(kr + d);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const float4 a = *reinterpret_cast<const float4*>(qw_rows + r * D + d);
        dot[r] = fmaf(a.x, c.x, dot[r]);
        dot[r] = fmaf(a.y, c.y, dot[r]);
        dot[r] = fmaf(a.z, c.z, dot[r]);
        dot[r] = fmaf(a.w, c.w, dot[r]);
      }
    }
    // levels 1-2 per row: running max and sum in base 2, the output rescaled
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qi = q0 + warp * kRowsPerWarp + r;
      const bool visible = key < Nk && (!causal || key <= qi) && (window <= 0 || key > qi - window);
      const float s2 = visible ? fmaf(slope2, static_cast<float>(key - qi), dot[r] * sl2) : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(s2));
      const float m_use = m_new == -INFINITY ? 0.f : m_new;  // no visible key for this row yet
      const float alpha = exp2f(m[r] - m_use);                 // 0 when m was -inf
      const float p = exp2f(s2 - m_use);                       // 0 for masked keys
      l[r] = fmaf(l[r], alpha, warp_sum(p));
#pragma unroll
      for (int c = 0; c < DC; ++c) acc[r][c] *= alpha;
      m[r] = m_new;
      pw[r * kBN + lane] = p;
    }
    __syncwarp();
    // level 3: acc += P V, four keys of every row per broadcast load
    for (int j = 0; j < kBN; j += 4) {
      float4 pr[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) pr[r] = *reinterpret_cast<const float4*>(pw + r * kBN + j);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float* vr = Vs + (j + jj) * D;
#pragma unroll
        for (int c = 0; c < DC; ++c) {
          const int d = lane + 32 * c;
          const float vv = d < D ? vr[d] : 0.f;
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            const float pj = jj == 0 ? pr[r].x : (jj == 1 ? pr[r].y : (jj == 2 ? pr[r].z : pr[r].w));
            acc[r][c] = fmaf(pj, vv, acc[r][c]);
          }
        }
      }
    }
    __syncwarp();  // the warp has read its probabilities before the next tile writes them
  }

  constexpr float kLn2 = 0.6931471805599453f;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int qi = q0 + warp * kRowsPerWarp + r;
    if (qi >= Nq) continue;
    const long long orow = (static_cast<long long>(b) * Hq + h) * Nq + qi;
    const bool live = l[r] > 0.f;
    const float inv = live ? 1.0f / l[r] : 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
      const int d = lane + 32 * c;
      if (d < D) o[orow * D + d] = acc[r][c] * inv;
    }
    if (lse && lane == 0) lse[orow] = live ? (m[r] + log2f(l[r])) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int D, float scale, int causal, int window, const float* alibi,
                            unsigned* status, cudaStream_t s) {
  const dim3 grid((Nq + kBM - 1) / kBM, Hq, B);
  if (B > 65535 || Hq > 65535) return cudaErrorInvalidConfiguration;
  const size_t smem = sizeof(float) * (kBM * D + kBN * (D + 4) + kBN * D + kWarps * kRowsPerWarp * kBN);
  const int dc = (D + 31) / 32;
  switch (dc) {
    case 1: attn_f32_kernel<1><<<grid, kWarps * 32, smem, s>>>(q, k, v, o, lse, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, status); break;
    case 2: attn_f32_kernel<2><<<grid, kWarps * 32, smem, s>>>(q, k, v, o, lse, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, status); break;
    case 3: attn_f32_kernel<3><<<grid, kWarps * 32, smem, s>>>(q, k, v, o, lse, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, status); break;
    default: attn_f32_kernel<4><<<grid, kWarps * 32, smem, s>>>(q, k, v, o, lse, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, status); break;
  }
  return cudaGetLastError();
}

}  // namespace rf
