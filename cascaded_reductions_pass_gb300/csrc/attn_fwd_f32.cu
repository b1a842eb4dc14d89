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
// this path uses FFMA throughout with the accurate exp2f/log2f.
//
// CTA: 64 query rows, 8 warps in two groups of 4.  The CTA's key tiles are
// split in two contiguous halves, one per group (the split of RedFuser's
// Figure 13, inside the CTA): warp w takes rows 16 (w mod 4) .. + 15 over
// the keys of group w / 4, and the two groups' (m, l, acc) states are merged
// once at the end.  Both products are register-tiled micro-GEMMs: lane =
// 8 rg + g (row group rg < 4, column group g < 8) holds rows rg + 4i (i < 4)
// of its warp, and
//   S = Q K^T   the keys g + 8i' (i' < 4) of the tile: 16 scores per lane,
//               32 packed fma.f32x2 (64 products) per four Q and four K
//               float4 loads;
//   O += P V    the output columns 4g + 32c + e (c < NC, e < 4): 16 NC
//               accumulators, 16 NC FFMA per key from one P and NC V float4.
// Row max and row sum finish with three shuffles inside the 8-lane group.
// Each group double-buffers its K and V tiles in shared memory by cp.async
// (the next tile streams in while the current one is used) and synchronises
// on a named barrier of its own; K and Q rows are padded to
// a stride of 4 (mod 32) words and P rows to 40 words, so every shared-memory
// access of a warp is conflict-free.  Exponentials are base 2 (log2 e folded
// into the scale) through exp2f, accurate to 2 ulp.  With the causal mask a
// sliding window (key j visible to query i iff i - window < j) and ALiBi
// biases (+ slope_h * (j - i)) are supported as in the tensor-core path.
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kGroupWarps = 4;           // warps per key group
constexpr int kGroups = 2;               // key groups per CTA
constexpr int kWarps = kGroupWarps * kGroups;
constexpr int kRowsW = 16;               // query rows per warp
constexpr int kBM = kGroupWarps * kRowsW;  // 64 query rows per CTA
constexpr int kBN = 32;                  // keys per tile
constexpr int kPS = 40;                  // P row stride (words)

__host__ __device__ __forceinline__ int padded_stride(int D) { return (D + 31) / 32 * 32 + 4; }

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void group_barrier(int id) {  // the 128 threads of one key group
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGroupWarps * 32) : "memory");
}

__device__ __forceinline__ float group_max(float v) {  // over the 8 lanes of a row group
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
}
__device__ __forceinline__ float group_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v + __shfl_xor_sync(0xffffffffu, v, 4);
}

// NC = ceil(D / 32): float4 output groups per lane.  DC: the head dimension
// fixed at compile time (so that every shared-memory offset is an immediate
// and the loops over D unroll), or 0 for any D <= 32 NC.  Up to D = 64 two
// CTAs fit an SM's shared memory; the launch bound keeps the registers to
// match (128 per thread).
template <int NC, int DC>
__global__ void __launch_bounds__(kWarps * 32, NC <= 2 ? 2 : 1) attn_f32_kernel(const float* __restrict__ q,
                                                               const float* __restrict__ k,
                                                               const float* __restrict__ v, float* __restrict__ o,
                                                               float* __restrict__ lse, int Hq, int Hkv, int Nq,
                                                               int Nk, int Dn, float scale, int causal, int window,
                                                               const float* __restrict__ alibi, unsigned* status) {
  static_assert(DC == 0 || (DC % 4 == 0 && DC <= 32 * NC && DC > 32 * (NC - 1)), "DC must match NC");
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  const int D = DC ? DC : Dn;
  const int KS = padded_stride(D);  // Q and K row stride (words)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / kGroupWarps, wr = warp % kGroupWarps;  // key group; row block of the warp
  const int gtid = threadIdx.x % (kGroupWarps * 32);            // thread index within the group
  const int rg = lane >> 3, g = lane & 7;
  float* Qs = smem;                                 // [kBM][KS]
  float* Ks = Qs + kBM * KS + grp * (2 * kBN * KS);  // this group's [2][kBN][KS]
  float* Vs = Qs + kBM * KS + kGroups * 2 * kBN * KS + grp * (2 * kBN * D);  // this group's [2][kBN][D]
  float* Ps = Qs + kBM * KS + kGroups * 2 * kBN * (KS + D);  // [kWarps][kRowsW][kPS]
  const int b = blockIdx.z, h = blockIdx.y, hk = h / (Hq / Hkv);
  const int q0 = blockIdx.x * kBM;
  // the grid is (query blocks, Hq, B): a block past them has nothing to do
  if (!RF_INB(q0 < Nq && h < Hq && hk < Hkv && D <= 32 * NC && (D & 3) == 0 && Dn == D, status)) return;
  const float* qh = q + (static_cast<long long>(b) * Hq + h) * Nq * D;
  const float* kh = k + (static_cast<long long>(b) * Hkv + hk) * Nk * D;
  const float* vh = v + (static_cast<long long>(b) * Hkv + hk) * Nk * D;
  const int D4 = D >> 2;
  constexpr float kLog2e = 1.4426950408889634f;
  const float sl2 = scale * kLog2e;  // scores in base-2 units

  const int last_row = min(q0 + kBM, Nq) - 1;
  const int kend = causal ? min(Nk, last_row + 1) : Nk;  // keys past the CTA's last row are all masked
  // a sliding window hides every key below the first row's window
  const int kbeg = (causal && window > 0) ? (max(0, q0 - window + 1) / kBN) * kBN : 0;
  const int ntiles_cta = kend > kbeg ? (kend - kbeg + kBN - 1) / kBN : 0;
  // group 0 takes the first ceil(n / 2) tiles, group 1 the rest
  const int n0 = (ntiles_cta + 1) / 2;
  const int tbeg = grp == 0 ? 0 : n0;
  const int ntiles = grp == 0 ? n0 : ntiles_cta - n0;
  const int bar_id = 1 + grp;  // the group's named barrier (barrier 0 is __syncthreads)

  // K and V rows [k0, k0 + kBN) into buffer `buf`; rows past Nk are zero-filled
  auto load_tile = [&](int k0, int buf) {
    float* kd = Ks + buf * kBN * KS;
    float* vd = Vs + buf * kBN * D;
    for (int i = gtid; i < kBN * D4; i += kGroupWarps * 32) {
      const int r = i / D4, c = i - r * D4;
      const bool ok = k0 + r < Nk;
      const long long src = static_cast<long long>(ok ? k0 + r : 0) * D + 4 * c;
      cp_async16(kd + r * KS + 4 * c, kh + src, ok);
      cp_async16(vd + r * D + 4 * c, vh + src, ok);
    }
  };
  for (int i = threadIdx.x; i < kBM * D4; i += kWarps * 32) {
    const int r = i / D4, c = i - r * D4;
    const bool ok = q0 + r < Nq;
    cp_async16(Qs + r * KS + 4 * c, qh + static_cast<long long>(ok ? q0 + r : 0) * D + 4 * c, ok);
  }
  cp_async_commit();
  if (ntiles > 0) load_tile(kbeg + tbeg * kBN, 0);
  cp_async_commit();
  cp_async_wait<1>();  // this thread's Q rows have landed
  __syncthreads();     // every thread's have

  float m[4], l[4], acc[4][NC][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][c][e] = 0.f;
  }
  const float slope2 = alibi ? __ldg(alibi + h) * kLog2e : 0.f;
  const float* qw = Qs + (wr * kRowsW + rg) * KS;  // row rg + 4i at qw + 4i KS
  float* pw = Ps + warp * kRowsW * kPS;
  const int row0 = q0 + wr * kRowsW + rg;          // query index of row i: row0 + 4i

  for (int t = 0; t < ntiles; ++t) {
    const int k0 = kbeg + (tbeg + t) * kBN, buf = t & 1;
    if (t + 1 < ntiles) load_tile(k0 + kBN, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // everything but the group just committed has landed
    group_barrier(bar_id);

    // S = Q K^T: rows rg + 4i, keys g + 8j of the tile.  Each score keeps two
    // partial sums, of its even and of its odd dimensions, as one packed pair:
    // (x, y) and (z, w) of a float4 are register pairs, so one fma.f32x2 does
    // two of the products.
    const float* kt = Ks + buf * kBN * KS + g * KS;
    uint64_t s2[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s2[i][j] = 0;
#pragma unroll
    for (int d = 0; d < D; d += 4) {
      ulonglong2 a[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const ulonglong2*>(qw + 4 * i * KS + d);
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = *reinterpret_cast<const ulonglong2*>(kt + 8 * j * KS + d);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s2[i][j] = fma_f32x2(a[i].x, c[j].x, s2[i][j]);
          s2[i][j] = fma_f32x2(a[i].y, c[j].y, s2[i][j]);
        }
    }
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo, hi;
        f2unpack(s2[i][j], lo, hi);
        s[i][j] = lo + hi;
      }
    // levels 1-2 per row: running max and sum in base 2, the output rescaled.
    // A tile whose keys every row of the warp sees needs no per-key test.
    const int wq0 = row0 - rg, wq1 = wq0 + kRowsW - 1;  // the warp's first and last query rows
    const bool interior = k0 + kBN <= Nk && (!causal || k0 + kBN - 1 <= wq0) && (window <= 0 || k0 > wq1 - window);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qi = row0 + 4 * i;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + g + 8 * j;
        const bool visible =
            interior || (key < Nk && (!causal || key <= qi) && (window <= 0 || key > qi - window));
        s[i][j] = visible ? fmaf(slope2, static_cast<float>(key - qi), s[i][j] * sl2) : -INFINITY;
        mx = fmaxf(mx, s[i][j]);
      }
      const float m_new = fmaxf(m[i], group_max(mx));
      const float m_use = m_new == -INFINITY ? 0.f : m_new;  // no visible key for this row yet
      const float alpha = exp2f(m[i] - m_use);                 // 0 when m was -inf
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = exp2f(s[i][j] - m_use);  // 0 for masked keys
        ps += p;
        pw[(rg + 4 * i) * kPS + g + 8 * j] = p;
      }
      l[i] = fmaf(l[i], alpha, group_sum(ps));
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][c][e] *= alpha;
      m[i] = m_new;
    }
    __syncwarp();
    // level 3: acc += P V over the tile's keys, four at a time
    const float* vt = Vs + buf * kBN * D;
    for (int j = 0; j < kBN; j += 4) {
      float4 pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = *reinterpret_cast<const float4*>(pw + (rg + 4 * i) * kPS + j);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float* vr = vt + (j + jj) * D;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int d = 4 * g + 32 * c;
          const float4 vv = d < D ? *reinterpret_cast<const float4*>(vr + d) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float pj = jj == 0 ? pr[i].x : (jj == 1 ? pr[i].y : (jj == 2 ? pr[i].z : pr[i].w));
            acc[i][c][0] = fmaf(pj, vv.x, acc[i][c][0]);
            acc[i][c][1] = fmaf(pj, vv.y, acc[i][c][1]);
            acc[i][c][2] = fmaf(pj, vv.z, acc[i][c][2]);
            acc[i][c][3] = fmaf(pj, vv.w, acc[i][c][3]);
          }
        }
      }
    }
    group_barrier(bar_id);  // the group is done with this buffer before the next prefetch overwrites it
  }
  cp_async_wait<0>();

  // Merge the two key groups (RedFuser, Figure 13): group 1 leaves its state
  // in its own K / V buffers and P rows, lane for lane; group 0 combines
  // m = max(m0, m1), l = l0 a0 + l1 a1, acc = acc0 a0 + acc1 a1 with
  // a_g = 2^(m_g - m).
  float* xacc = Qs + kBM * KS + 2 * kBN * KS;  // group 1's K buffers: [4 warps][32 lanes][4][NC][4]
  float* xml = Ps + kGroupWarps * kRowsW * kPS;  // group 1's P rows: [4 warps][32 lanes][8]
  if (grp == 1) {
    float* xa = xacc + (wr * 32 + lane) * (16 * NC);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < NC; ++c)
        *reinterpret_cast<float4*>(xa + (i * NC + c) * 4) =
            make_float4(acc[i][c][0], acc[i][c][1], acc[i][c][2], acc[i][c][3]);
    float* xm = xml + (wr * 32 + lane) * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xm[i] = m[i];
      xm[4 + i] = l[i];
    }
  }
  __syncthreads();
  if (grp == 1) return;
  {
    const float* xa = xacc + (wr * 32 + lane) * (16 * NC);
    const float* xm = xml + (wr * 32 + lane) * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float m1 = xm[i], l1 = xm[4 + i];
      const float mm = fmaxf(m[i], m1);
      const float mu = mm == -INFINITY ? 0.f : mm;
      const float a0 = exp2f(m[i] - mu), a1 = exp2f(m1 - mu);
      l[i] = l[i] * a0 + l1 * a1;
      m[i] = mm;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(xa + (i * NC + c) * 4);
        acc[i][c][0] = fmaf(acc[i][c][0], a0, x.x * a1);
        acc[i][c][1] = fmaf(acc[i][c][1], a0, x.y * a1);
        acc[i][c][2] = fmaf(acc[i][c][2], a0, x.z * a1);
        acc[i][c][3] = fmaf(acc[i][c][3], a0, x.w * a1);
      }
    }
  }

  constexpr float kLn2 = 0.6931471805599453f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qi = row0 + 4 * i;
    if (qi >= Nq) continue;
    const long long orow = (static_cast<long long>(b) * Hq + h) * Nq + qi;
    const bool live = l[i] > 0.f;
    const float inv = live ? 1.0f / l[i] : 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = 4 * g + 32 * c;
      if (d < D)
        *reinterpret_cast<float4*>(o + orow * D + d) =
            make_float4(acc[i][c][0] * inv, acc[i][c][1] * inv, acc[i][c][2] * inv, acc[i][c][3] * inv);
    }
    if (lse && g == 0) lse[orow] = live ? (m[i] + log2f(l[i])) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int D, float scale, int causal, int window, const float* alibi,
                            unsigned* status, cudaStream_t s) {
  const dim3 grid((Nq + kBM - 1) / kBM, Hq, B);
  if (B > 65535 || Hq > 65535) return cudaErrorInvalidConfiguration;
  const int KS = padded_stride(D);
  const size_t smem =
      sizeof(float) * (static_cast<size_t>(kBM) * KS + kGroups * 2 * kBN * (KS + D) + kWarps * kRowsW * kPS);
  const int nc = (D + 31) / 32;
  const bool fixed = D == 32 * nc;  // 32, 64, 96, 128: the compile-time instances
#define RF_F32_LAUNCH(NC, DC)                                                                               \
  do {                                                                                                      \
    cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<NC, DC>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                         static_cast<int>(smem));                                           \
    if (e != cudaSuccess) return e;                                                                         \
    attn_f32_kernel<NC, DC><<<grid, kWarps * 32, smem, s>>>(q, k, v, o, lse, Hq, Hkv, Nq, Nk, D, scale, causal, \
                                                            window, alibi, status);                         \
  } while (0)
  switch (nc) {
    case 1: if (fixed) RF_F32_LAUNCH(1, 32); else RF_F32_LAUNCH(1, 0); break;
    case 2: if (fixed) RF_F32_LAUNCH(2, 64); else RF_F32_LAUNCH(2, 0); break;
    case 3: if (fixed) RF_F32_LAUNCH(3, 96); else RF_F32_LAUNCH(3, 0); break;
    default: if (fixed) RF_F32_LAUNCH(4, 128); else RF_F32_LAUNCH(4, 0); break;
  }
#undef RF_F32_LAUNCH
  return cudaGetLastError();
}

}  // namespace rf
