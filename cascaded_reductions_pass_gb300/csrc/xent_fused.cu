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
//
// Few rows (a decoding step's last-token logits): one CTA per row would leave
// most SMs idle and run at one SM's load latency, so a thread-block cluster of
// up to 8 CTAs takes each row instead.  Each CTA folds its slice of the
// vocabulary into a running (m, l); rank 0 of the cluster merges the CTAs'
// pairs, read from their shared memory through the cluster's distributed
// shared memory, with the same log-sum-exp combine (the split-vocabulary
// merge), writes loss and LSE, and hands the LSE back to every CTA for the
// gradient pass over its own slice.  No workspace is involved.
#include <cooperative_groups.h>
#include <math.h>

#include "rf_device.cuh"

namespace cg = cooperative_groups;

namespace rf {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;
// Below this many 16-byte vectors per row (e.g. a 32000-entry bf16 vocabulary:
// 4000), one row per 256-thread CTA streams 23% faster than per 512-thread CTA
// (measured at 8192 rows); from 128256 entries on, 512 threads are as fast or
// faster.
constexpr int kShortRowVecs = 8192;
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
  // the block max by 3-input maxima
  float bm;
  if constexpr (E == 8) {
    bm = fmaxf(max3f(z[0], z[1], z[2]), max3f(z[3], z[4], max3f(z[5], z[6], z[7])));
  } else {
    static_assert(E == 4, "16-byte blocks of 2- or 4-byte elements");
    bm = fmaxf(max3f(z[0], z[1], z[2]), z[3]);
  }
  bm *= kLog2e;
  if (bm > r.m) {  // level 1 moved: correct level 2 by 2^(m_old - m_new)
    r.l *= ex2_ftz(r.m - bm);
    r.m = bm;
  }
  if (r.m == -INFINITY) return;  // nothing finite seen yet (all -inf logits)
  // exponent arguments and the partial sum on packed pairs
  const uint64_t l2 = f2pack(kLog2e, kLog2e), nm2 = f2pack(-r.m, -r.m);
  uint64_t s2 = 0;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    float x0, x1;
    f2unpack(fma_f32x2(f2pack(z[e], z[e + 1]), l2, nm2), x0, x1);
    s2 = add_f32x2(s2, f2pack(ex2_ftz(x0), ex2_ftz(x1)));
  }
  float lo, hi;
  f2unpack(s2, lo, hi);
  r.l += lo + hi;
}

// This thread's running (m, l) over the row's 16-byte vectors [c0, c1).
// Every pass issues its (up to) four loads before folding any, also at the
// end of a slice, so a short slice costs one load latency, not four.
template <Dt DT, int NT>
__device__ __forceinline__ Run fold_range(const uint4* __restrict__ zr, int c0, int c1) {
  Run run{-INFINITY, 0.f};
  for (int c = c0 + threadIdx.x; c < c1; c += kUnroll * NT) {
    uint4 u[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (c + k * NT < c1) u[k] = ld_stream(zr + c + k * NT);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (c + k * NT < c1) fold_block<DT>(u[k], run);
  }
  return run;
}

// Merge the CTA's NT threads: warp shuffles, then the warps in shared memory.
template <int NT>
__device__ __forceinline__ Run cta_combine(Run run, Run* s_run) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Run b{__shfl_xor_sync(0xffffffffu, run.m, o), __shfl_xor_sync(0xffffffffu, run.l, o)};
    run = lse_combine(run, b);
  }
  if ((tid & 31) == 0) s_run[tid >> 5] = run;
  __syncthreads();
  run = s_run[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) run = lse_combine(run, s_run[w]);
  return run;
}

// loss of one row from its LSE (natural log): 0 if ignored, NaN for a target
// outside [0, V), else lse - z[target]
template <Dt DT>
__device__ __forceinline__ float row_loss(const uint4* __restrict__ logits, long long row, long long V, long long t,
                                          long long ignore_index, float lse) {
  if (t == ignore_index) return 0.f;
  if (t < 0 || t >= V) return __int_as_float(0x7fc00000);
  const uint16_t* z16 = reinterpret_cast<const uint16_t*>(logits);
  float zt;
  if constexpr (DT == Dt::F32)
    zt = reinterpret_cast<const float*>(logits)[row * V + t];
  else if constexpr (DT == Dt::BF16)
    zt = __uint_as_float(static_cast<uint32_t>(z16[row * V + t]) << 16);
  else
    zt = __half2float(__ushort_as_half(z16[row * V + t]));
  return lse - zt;
}

// gradient softmax(z) - onehot(t) over vectors [c0, c1), or 0 for an ignored row
template <Dt DT, int NT>
__device__ __forceinline__ void write_grad(const uint4* __restrict__ zr, uint4* __restrict__ gr, int c0, int c1,
                                           float lse2, long long t, bool ignored) {
  constexpr int E = Pack<DT>::E;
  for (int c = c0 + threadIdx.x; c < c1; c += kUnroll * NT) {
    uint4 u[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k)
      if (!ignored && c + k * NT < c1) u[k] = __ldg(zr + c + k * NT);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int cc = c + k * NT;
      if (cc >= c1) continue;
      float g[E];
      if (ignored) {
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = 0.f;
      } else {
        float z[E];
        Pack<DT>::unpack(u[k], z);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          g[e] = ex2_ftz(fmaf(z[e], kLog2e, -lse2));
          if (static_cast<long long>(cc) * E + e == t) g[e] -= 1.f;
        }
      }
      st_stream(gr + cc, Pack<DT>::pack(g));
    }
  }
}

// One CTA of NT threads per row.
template <Dt DT, int NT>
__global__ void __launch_bounds__(NT) xent_kernel(const uint4* __restrict__ logits,
                                                  const long long* __restrict__ targets,
                                                  float* __restrict__ loss, float* __restrict__ lse_out,
                                                  uint4* __restrict__ grad, int nvec, long long ignore_index,
                                                  int rows, unsigned* status) {
  constexpr int E = Pack<DT>::E;
  __shared__ Run s_run[NT / 32];
  const long long row = blockIdx.x;
  if (!RF_INB(row < rows, status)) return;
  const uint4* zr = logits + row * nvec;
  const Run run = cta_combine<NT>(fold_range<DT, NT>(zr, 0, nvec), s_run);
  const float lse2 = run.m + log2f(run.l);  // base 2
  const float lse = lse2 * kLn2;
  const long long t = targets[row];
  const long long V = static_cast<long long>(nvec) * E;
  if (threadIdx.x == 0) {
    if (lse_out) lse_out[row] = lse;
    loss[row] = row_loss<DT>(logits, row, V, t, ignore_index, lse);
  }
  if (grad) write_grad<DT, NT>(zr, grad + row * nvec, 0, nvec, lse2, t, t == ignore_index);
}

// One row per cluster of `cs` CTAs (cluster rank = slice of the vocabulary).
template <Dt DT>
__global__ void __launch_bounds__(kThreads) xent_cluster_kernel(const uint4* __restrict__ logits,
                                                                const long long* __restrict__ targets,
                                                                float* __restrict__ loss,
                                                                float* __restrict__ lse_out,
                                                                uint4* __restrict__ grad, int nvec,
                                                                long long ignore_index, int rows,
                                                                unsigned* status) {
  constexpr int E = Pack<DT>::E;
  __shared__ Run s_run[kThreads / 32];
  __shared__ Run s_part;   // this CTA's (m, l), read by rank 0
  __shared__ float s_lse2; // the row's LSE (base 2), written by rank 0
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const long long row = blockIdx.x / cs;
  const int c0 = static_cast<int>(static_cast<long long>(nvec) * rank / cs);
  const int c1 = static_cast<int>(static_cast<long long>(nvec) * (rank + 1) / cs);
  // every CTA of the cluster meets the cluster barriers below, so a failed
  // check only empties its slice
  const bool in_row = RF_INB(row < rows && c0 >= 0 && c0 <= c1 && c1 <= nvec, status);
  const uint4* zr = logits + (in_row ? row : 0) * nvec;
  const Run part = cta_combine<kThreads>(fold_range<DT, kThreads>(zr, in_row ? c0 : 0, in_row ? c1 : 0), s_run);
  if (threadIdx.x == 0) s_part = part;
  cluster.sync();  // every slice's (m, l) is in its CTA's shared memory
  if (rank == 0 && threadIdx.x == 0 && in_row) {
    Run run = s_part;
    for (int r = 1; r < cs; ++r) run = lse_combine(run, *cluster.map_shared_rank(&s_part, r));
    const float lse2 = run.m + log2f(run.l);
    for (int r = 0; r < cs; ++r) *cluster.map_shared_rank(&s_lse2, r) = lse2;
    const float lse = lse2 * kLn2;
    const long long t = targets[row];
    if (lse_out) lse_out[row] = lse;
    loss[row] = row_loss<DT>(logits, row, static_cast<long long>(nvec) * E, t, ignore_index, lse);
  }
  cluster.sync();  // s_lse2 is set everywhere; no CTA reads another's shared memory after this
  if (grad && in_row) {
    const long long t = targets[row];
    write_grad<DT, kThreads>(zr, grad + row * nvec, c0, c1, s_lse2, t, t == ignore_index);
  }
}

// Cluster size for `rows` rows: enough CTAs for one per SM, at most 8 (the
// portable cluster size), and at least 512 vectors (one full pass of the
// CTA) per CTA; 1 means one CTA per row.
int xent_cluster_size(int rows, int nvec, int sms) {
  int cs = 1;
  while (cs < 8 && static_cast<long long>(rows) * cs < sms && nvec / (2 * cs) >= kThreads) cs *= 2;
  return cs;
}

template <Dt DT>
cudaError_t launch_dt(const uint4* L, const long long* targets, float* loss, float* lse, uint4* G, int rows,
                      int nvec, long long ignore_index, int sms, unsigned* status, cudaStream_t s) {
  const int cs = xent_cluster_size(rows, nvec, sms);
  if (cs == 1) {
    // rows of fewer than kShortRowVecs vectors: CTAs of half the size (more rows in flight per SM)
    if (nvec < kShortRowVecs)
      xent_kernel<DT, kThreads / 2><<<rows, kThreads / 2, 0, s>>>(L, targets, loss, lse, G, nvec, ignore_index, rows,
                                                                   status);
    else
      xent_kernel<DT, kThreads><<<rows, kThreads, 0, s>>>(L, targets, loss, lse, G, nvec, ignore_index, rows, status);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows) * cs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, xent_cluster_kernel<DT>, L, targets, loss, lse, G, nvec, ignore_index, rows, status);
}

}  // namespace

cudaError_t launch_xent(const void* logits, const long long* targets, float* loss, float* lse, void* grad, int rows,
                        int vocab, long long ignore_index, Dt dt, unsigned* status, cudaStream_t s) {
  const int E = dt == Dt::F32 ? 4 : 8;
  const int nvec = vocab / E;
  const int sms = device_sm_count();
  auto L = static_cast<const uint4*>(logits);
  auto G = static_cast<uint4*>(grad);
  switch (dt) {
    case Dt::F32: return launch_dt<Dt::F32>(L, targets, loss, lse, G, rows, nvec, ignore_index, sms, status, s);
    case Dt::F16: return launch_dt<Dt::F16>(L, targets, loss, lse, G, rows, nvec, ignore_index, sms, status, s);
    case Dt::BF16: return launch_dt<Dt::BF16>(L, targets, loss, lse, G, rows, nvec, ignore_index, sms, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rf
