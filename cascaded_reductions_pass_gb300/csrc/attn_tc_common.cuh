// attn_tc_common.cuh -- constants and per-row softmax steps shared by the
// tensor-core attention kernels (attn_fwd_tc.cu, attn_fwd_tc_window.cu): the
// tile sizes, the warp layout and register split, the unit order, and the
// level-1 / level-2 steps of one row of a score tile.
#pragma once

#include "rf_device.cuh"

namespace rf {
namespace {

constexpr int kBM = 128;        // query rows per tile (TMEM lanes)
constexpr int kBN = 128;        // keys per tile
constexpr int kThreads = 384;   // 12 warps
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // base-2 units
constexpr int kRegsCtl = 80;       // per thread, warps 0-3 after reallocation
constexpr int kRegsSoftmax = 208;  // per thread, warps 4-11 after reallocation

// Unit (CTA of whole rows) id -> query-tile pair c and batch*head bh: the
// longest causal units first, the heads of one GQA group adjacent.
__host__ __device__ __forceinline__ void unit_coords(int id, int BH, int nqt, int& c, int& bh) {
  c = nqt - 1 - id / BH;
  bh = id - (id / BH) * BH;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Max of the scores s[C0, kBN) of a row, in the base-2 units of the exponent
// (ALiBi rows already hold scaled scores): independent 3-input max chains of
// 32 elements each.
template <int C0, bool ALIBI>
__device__ __forceinline__ float scaled_max_from(const uint32_t* s, float sl2) {
  constexpr int kChains = (kBN - C0) / 32;
  float mx[kChains];
#pragma unroll
  for (int q4 = 0; q4 < kChains; ++q4) {
    const uint32_t* sq = s + C0 + 32 * q4;
    float m = max3f(__uint_as_float(sq[0]), __uint_as_float(sq[1]), __uint_as_float(sq[2]));
#pragma unroll
    for (int i = 3; i + 1 < 32; i += 2) m = max3f(m, __uint_as_float(sq[i]), __uint_as_float(sq[i + 1]));
    mx[q4] = fmaxf(m, __uint_as_float(sq[31]));
  }
  float m = mx[0];
#pragma unroll
  for (int q4 = 1; q4 < kChains; ++q4) m = fmaxf(m, mx[q4]);
  return ALIBI ? m : m * sl2;
}

// P = 2^(s * sl2 - m) for the pairs [E0, E1) of a row (16-bit, packed into
// pk), and their sum, kept in four packed accumulators.
template <Dt DT, bool ALIBI, int E0, int E1>
__device__ __forceinline__ float exp_pairs(const uint32_t* s, uint64_t sl2x2, uint64_t negm2, uint32_t* pk) {
  uint64_t sum2[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) sum2[q4] = f2pack(0.f, 0.f);
#pragma unroll
  for (int e = E0; e < E1; ++e) {
    const uint64_t x = ALIBI ? add_f32x2(u2pack(s[2 * e], s[2 * e + 1]), negm2)
                             : fma_f32x2(u2pack(s[2 * e], s[2 * e + 1]), sl2x2, negm2);
    float x0, x1;
    f2unpack(x, x0, x1);
    const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
    sum2[e & 3] = add_f32x2(sum2[e & 3], f2pack(p0, p1));
    pk[e] = Pack<DT>::pack2(p0, p1);
  }
  float lo, hi;
  f2unpack(add_f32x2(add_f32x2(sum2[0], sum2[1]), add_f32x2(sum2[2], sum2[3])), lo, hi);
  return lo + hi;
}

// A packed pair of 16-bit P values times a.
template <Dt DT>
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float a) {
  float lo, hi;
  if constexpr (DT == Dt::BF16) {
    lo = bf16lo(w);
    hi = bf16hi(w);
  } else {
    const float2 f = unpack_f16x2(w);
    lo = f.x;
    hi = f.y;
  }
  return Pack<DT>::pack2(lo * a, hi * a);
}

}  // namespace
}  // namespace rf
