// decode_split.cu -- split-KV decoding: the per-split partial results.
//
// One decoding step attends one query per head to a KV cache of L keys
// (AttnFuse, Table 8 "Flash Decoding"; RedFuser, Figure 13 "FlashDecoding
// IR").  The keys of each (batch, kv head) are cut into S contiguous splits,
// split s covering [floor(s*L/S), floor((s+1)*L/S)); one CTA runs the fused
// cascade max -> sum exp -> sum exp*v over one split for all G = Hq/Hkv query
// heads that share the kv head, in the incremental form of RedFuser's
// Figure 4: per 64-key tile the running max per head is raised and the
// running sum and output are rescaled by exp(m_old - m_new).  The split's
// normalised O_s and lse_s = m + ln l go to the caller's workspace; the
// log-sum-exp merge (lse_merge.cu) combines the splits.
//
// Data path (HBM-bound: every K/V byte is read once):
//  * a producer warp streams 64-key tiles of K and V into a 3-stage ring of
//    shared memory with TMA (128-byte swizzle, 64 x 64 boxes), completion
//    tracked by mbarriers;
//  * four consumer warps each take 16 keys of every tile.  Scores are computed
//    transposed, S^T = K Q^T, with mma.sync m16n8k16 (M = 16 keys, N = 8 query
//    heads, K = 16 head dims): the 8 query heads of a group fill N exactly, so
//    no MMA row is padding.  P^T is turned into the B operand of O^T += V^T P^T
//    with movmatrix (an in-register 8x8 transpose) and V^T comes from
//    ldmatrix.trans, so O^T stays in registers (D x 8 per warp);
//  * at the end the four warps' (m, l, O) are merged through shared memory
//    with the same rescaling, and the split result is written.
// Each mbarrier wait is bounded; a wait that runs out sets the device status
// word, the CTA stops consuming, the producer waits for its copies in flight,
// the split's partials are written as NaN, and the kernel returns.
#include <cuda.h>
#include <math.h>

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kBN = 64;          // keys per tile
constexpr int kStages = 3;       // K/V ring depth
constexpr int kConsumers = 4;    // consumer warps (16 keys each per tile)
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <Dt DT>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (DT == Dt::BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Byte offset of (key r, 16-byte chunk c) inside one 64-key x 128-byte TMA box
// written with the 128-byte swizzle (chunk index XORed with r mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) { return uint32_t(r * 128 + ((c ^ (r & 7)) << 4)); }

struct alignas(8) Bars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

template <Dt DT, int D>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                        const uint16_t* __restrict__ q, float* __restrict__ o_part, float* __restrict__ lse_part,
                        int Hq, int Hkv, int L, int S, float scale_log2, unsigned* status) {
  constexpr int kBoxes = D / 64;                       // 64-dim boxes per key row
  constexpr int kTileBytes = kBN * D * 2;              // one tensor's tile
  constexpr int kStageBytes = 2 * kTileBytes;          // K + V
  constexpr int kDC = D / 16;                          // 16-wide head-dim chunks
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kStages * kStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const long long lo = (static_cast<long long>(split) * L) / S;
  const long long hi = (static_cast<long long>(split + 1) * L) / S;
  const int ntiles = static_cast<int>((hi - lo + kBN - 1) / kBN);
  const int plane = b * Hkv + hk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], kConsumers);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();  // the merge may be scheduled once every split has started

  // Per-lane partial state (consumer warps): heads 2t, 2t+1 of the group.
  const int g = lane >> 2, t = lane & 3;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float acc[kDC][4];
#pragma unroll
  for (int i = 0; i < kDC; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  if (warp == kConsumers) {
    // ---------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int issued = 0;
      for (int it = 0; it < ntiles; ++it) {
        const int st = it % kStages;
        if (it >= kStages && !mbar_wait(&bars->empty[st], ((it / kStages) - 1) & 1)) {
          atomicOr(status, kStatusTimeout);
          bars->abort = 1;
          break;
        }
        if (*reinterpret_cast<volatile int*>(&bars->abort)) break;
        uint8_t* dst = smem + st * kStageBytes;
        mbar_expect_tx(&bars->full[st], kStageBytes);
        const int key0 = static_cast<int>(lo) + it * kBN;
        (void)RF_INB(key0 < L && plane < static_cast<int>(gridDim.z) * Hkv, status);
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
          tma_load_3d(dst + bx * (kBN * 128), &tk, &bars->full[st], bx * 64, key0, plane);
          tma_load_3d(dst + kTileBytes + bx * (kBN * 128), &tv, &bars->full[st], bx * 64, key0, plane);
        }
        ++issued;
      }
      // Drain: every copy issued must land before the CTA may exit.
      for (int it = issued > kStages ? issued - kStages : 0; it < issued; ++it) {
        if (!mbar_wait(&bars->full[it % kStages], (it / kStages) & 1)) atomicOr(status, kStatusTimeout);
      }
    }
  } else {
    // ---------------- consumers
    // Q^T as the B operand: lane (g, t) holds head g's dims {16c+2t, +1} and {16c+2t+8, +9}.
    uint32_t qf[kDC][2];
    const int hq = hk * G + g;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q + (static_cast<long long>(b) * Hq + hq) * D);
    const bool q_in = g >= G || RF_INB(b < static_cast<int>(gridDim.z) && hq < Hq, status);
#pragma unroll
    for (int c = 0; c < kDC; ++c) {
      qf[c][0] = g < G && q_in ? __ldg(qrow + 8 * c + t) : 0u;
      qf[c][1] = g < G && q_in ? __ldg(qrow + 8 * c + 4 + t) : 0u;
    }
    const uint32_t smem_base = smem_u32(smem);
    // ldmatrix lane roles: K (non-transposed A) and V (transposed A) address maps.
    const int mi = lane >> 3, rr = lane & 7;
    const int k_key = warp * 16 + rr + 8 * (mi & 1), k_chunk = mi >> 1;  // key row, +8-dim half
    const int v_key = warp * 16 + rr + 8 * (mi >> 1), v_chunk = mi & 1;

    for (int it = 0; it < ntiles; ++it) {
      const int st = it % kStages;
      if (!mbar_wait(&bars->full[st], (it / kStages) & 1)) {
        atomicOr(status, kStatusTimeout);
        bars->abort = 1;
        break;
      }
      const uint32_t kbase = smem_base + st * kStageBytes;
      const uint32_t vbase = kbase + kTileBytes;

      // S^T (16 keys x 8 heads) = K_sub Q^T
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kDC; ++c) {
        const int box = c >> 2, ch = ((c & 3) << 1) + k_chunk;  // 16-byte chunk within the box row
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + box * (kBN * 128) + swz(k_key, ch), a0, a1, a2, a3);
        mma16816<DT>(s, a0, a1, a2, a3, qf[c][0], qf[c][1]);
      }
      // scale (log2 domain) and mask keys outside the split
      const long long key_a = lo + static_cast<long long>(it) * kBN + warp * 16 + g;
      const bool va = key_a < hi, vb = key_a + 8 < hi;
      s[0] = va ? s[0] * scale_log2 : -INFINITY;
      s[1] = va ? s[1] * scale_log2 : -INFINITY;
      s[2] = vb ? s[2] * scale_log2 : -INFINITY;
      s[3] = vb ? s[3] * scale_log2 : -INFINITY;
      // level 1: running max per head (reduce over the 16 keys: c0/c2 and lanes g)
      float tm0 = fmaxf(s[0], s[2]), tm1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, o));
        tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, o));
      }
      const float mn0 = fmaxf(m[0], tm0), mn1 = fmaxf(m[1], tm1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m[0] - mu0), al1 = exp2f(m[1] - mu1);
      m[0] = mn0;
      m[1] = mn1;
      // level 2: p = exp(s - m); running (per-lane partial) sums
      const float p0 = exp2f(s[0] - mu0), p1 = exp2f(s[1] - mu1), p2 = exp2f(s[2] - mu0), p3 = exp2f(s[3] - mu1);
      l[0] = fmaf(l[0], al0, p0 + p2);
      l[1] = fmaf(l[1], al1, p1 + p3);
      // P^T -> B operand of O^T += V^T P^T (8x8 transposes in registers)
      const uint32_t pb0 = movmatrix_t(Pack<DT>::pack2(p0, p1));
      const uint32_t pb1 = movmatrix_t(Pack<DT>::pack2(p2, p3));
      // level 3: rescale the running output, add this tile's terms
#pragma unroll
      for (int c = 0; c < kDC; ++c) {
        acc[c][0] *= al0;
        acc[c][1] *= al1;
        acc[c][2] *= al0;
        acc[c][3] *= al1;
        const int box = c >> 2, ch = ((c & 3) << 1) + v_chunk;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + box * (kBN * 128) + swz(v_key, ch), a0, a1, a2, a3);
        mma16816<DT>(acc[c], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[st]);
    }
  }
  __syncthreads();

  // ---------------- merge the four warps' partial results (shared memory reused)
  float* cm = reinterpret_cast<float*>(smem);      // [4][8] running max (log2 domain)
  float* cl = cm + kConsumers * 8;                  // [4][8] running sums
  float* co = cl + kConsumers * 8;                  // [4][8][D] running outputs
  if (warp < kConsumers) {
    float l0 = l[0], l1 = l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (g == 0) {
      cm[warp * 8 + 2 * t] = m[0];
      cm[warp * 8 + 2 * t + 1] = m[1];
      cl[warp * 8 + 2 * t] = l0;
      cl[warp * 8 + 2 * t + 1] = l1;
    }
#pragma unroll
    for (int c = 0; c < kDC; ++c) {
      const int d = 16 * c + g;
      co[(warp * 8 + 2 * t) * D + d] = acc[c][0];
      co[(warp * 8 + 2 * t + 1) * D + d] = acc[c][1];
      co[(warp * 8 + 2 * t) * D + d + 8] = acc[c][2];
      co[(warp * 8 + 2 * t + 1) * D + d + 8] = acc[c][3];
    }
  }
  __syncthreads();
  if (bars->abort) {
    // A wait gave up: mark this split's partials invalid (NaN), so that the
    // merge turns the rows into NaN instead of combining stale slots.
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int h = idx / D, d = idx - h * D;
      const long long row = static_cast<long long>(b) * Hq + hk * G + h;
      if (!RF_INB(row < static_cast<long long>(gridDim.z) * Hq && split < S, status)) continue;
      o_part[(row * S + split) * D + d] = NAN;
      if (d == 0) lse_part[row * S + split] = NAN;
    }
    return;
  }
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, cm[w * 8 + h]);
    const long long row = static_cast<long long>(b) * Hq + hk * G + h;
    float out = 0.f, lse = -INFINITY;
    if (M != -INFINITY) {
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float f = exp2f(cm[w * 8 + h] - M);
        num = fmaf(f, co[(w * 8 + h) * D + d], num);
        den = fmaf(f, cl[w * 8 + h], den);
      }
      out = num / den;
      lse = (M + log2f(den)) * kLn2;
    }
    if (!RF_INB(row < static_cast<long long>(gridDim.z) * Hq && split < S, status)) continue;
    o_part[(row * S + split) * D + d] = out;
    if (d == 0) lse_part[row * S + split] = lse;
  }
}

template <Dt DT, int D>
cudaError_t launch_dt(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int Hq,
                      int Hkv, int L, int S, float scale, unsigned* status, cudaStream_t s) {
  alignas(64) CUtensorMap tk, tv;
  cudaError_t err = cudaSuccess;
  if (!encode_tma_3d_16bit(&tk, k, D, L, uint64_t(B) * Hkv, kBN, &err)) return err;
  if (!encode_tma_3d_16bit(&tv, v, D, L, uint64_t(B) * Hkv, kBN, &err)) return err;
  constexpr int kSmem = kStages * 2 * kBN * D * 2 + 1024 + 128;
  static_assert(kStages * 2 * kBN * D * 2 >= (8 * 4 * 2 + 32 * D) * 4, "merge buffer must fit in the ring");
  auto kern = decode_split_kernel<DT, D>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  if (Hkv > 65535 || B > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(S, Hkv, B);
  kern<<<grid, kThreads, kSmem, s>>>(tk, tv, static_cast<const uint16_t*>(q), o_part, lse_part, Hq, Hkv, L, S,
                                     scale * kLog2e, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_split(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B,
                                int Hq, int Hkv, int L, int D, int splits, float scale, Dt dt, unsigned* status,
                                cudaStream_t s) {
  if (dt == Dt::BF16) {
    return D == 128 ? launch_dt<Dt::BF16, 128>(q, k, v, o_part, lse_part, B, Hq, Hkv, L, splits, scale, status, s)
                    : launch_dt<Dt::BF16, 64>(q, k, v, o_part, lse_part, B, Hq, Hkv, L, splits, scale, status, s);
  }
  if (dt == Dt::F16) {
    return D == 128 ? launch_dt<Dt::F16, 128>(q, k, v, o_part, lse_part, B, Hq, Hkv, L, splits, scale, status, s)
                    : launch_dt<Dt::F16, 64>(q, k, v, o_part, lse_part, B, Hq, Hkv, L, splits, scale, status, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace rf
