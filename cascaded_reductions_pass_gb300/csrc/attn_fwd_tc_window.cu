// attn_fwd_tc_window.cu -- causal sliding-window attention on the tensor cores
// for fp16/bf16 inputs at D = 64, as a persistent kernel.
//
// The cascade, tiles, warp roles, TMEM layout and per-key-tile steps are those
// of attn_fwd_tc.cu at D = 64 (P in TMEM columns of its own, so S_t(j+1) is
// issued while softmax t still exponentiates tile j).  What differs is the
// schedule.  With a window of W keys, a unit of 256 query rows touches only
// about (W + 256) / 128 key tiles, so a CTA per unit would spend much of its
// time on fixed costs: TMEM allocation, barrier setup, loading Q, filling and
// draining the pipeline, the epilogue.  Here one CTA per SM walks a list of
// units (its work items), and those costs overlap the neighbouring units' work:
//  * Q is double-buffered: item k+1's two query tiles load while item k runs;
//  * the K/V rings and every barrier's phase run on across items, so the ring
//    never drains between items;
//  * the MMA issuer issues item k+1's first S as soon as softmax has read item
//    k's last S, so the next item's first exponentials overlap item k's last
//    PV and its epilogue.
// Dense and plain causal attention keep one CTA per unit: wrapping the MMA
// issuer's key-tile loop in a loop over items was measured to lengthen its
// per-tile steps by about 10%, which units of 16-32 key tiles never win back.
//
// Work items: the units in the order of unit_coords; CTA b of a grid of G takes
// item k*G + b in even rounds k and k*G + G-1-b in odd ones.  The item table is
// built in shared memory before the register split (its integer divisions
// inside the 80-register issuer region slowed the issue loop).
// Every mbarrier wait is bounded; on a timeout the CTA records RF_ERR_TIMEOUT,
// tells its other warps to stop at the next item, waits (bounded) for its
// copies and MMAs in flight, frees TMEM and exits.
#include <cuda.h>
#include <math.h>

#include "attn_tc_common.cuh"
#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kWD = 64;                      // head dimension
constexpr int kWQBytes = kBM * kWD * 2;      // one query tile
constexpr int kWKVBytes = kBN * kWD * 2;     // one K or V tile
constexpr int kWStages = 3;                  // K/V ring depth
constexpr int kWTiles = 2 * 2 * kWQBytes + 2 * kWStages * kWKVBytes;  // Q [tile][buffer], K ring, V ring
constexpr int kWOStage = 8 * 32 * kWD * 2;   // O staging: 32 rows x 128 B per softmax warp
constexpr int kWOCol = 2 * kBN;              // O0 at 256, O1 at 320
constexpr int kWPCol = 2 * kBN + 2 * kWD;    // P0 at 384, P1 at 448
constexpr int kMaxItems = 1024;              // items per CTA (the grid widens beyond that)

struct alignas(8) WinBars {
  uint64_t q_full[2][2], q_empty[2][2];  // [query tile][Q buffer]
  uint64_t k_full[kWStages], k_empty[kWStages], v_full[kWStages], v_empty[kWStages];
  uint64_t s_full[2], s_free[2], p_ready[2], pv_done[2], o_final[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// One work item: a unit of 256 query rows (rows r0..r0+255 of plane bh) and the
// key tiles [lo_t, nt_t) that its query tile t sees (lo0 <= lo1, nt0 <= nt1).
// Tile 0's range is never empty (Nq == Nk); tile 1's is empty when all its rows
// lie past Nq.  bh < 0 ends a CTA's list.
struct WinItem {
  int bh, r0, lo0, nt0, lo1, nt1;
};

struct WinSched {
  int BH, nqt, Nk, window, n_items;
};

__device__ __forceinline__ bool win_item(const WinSched& sc, int k, WinItem& it) {
  const int G = gridDim.x, b = blockIdx.x;
  const long long i = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - b : b);
  if (i >= sc.n_items) return false;
  int c;
  unit_coords(static_cast<int>(i), sc.BH, sc.nqt, c, it.bh);
  it.r0 = c * 2 * kBM;
  const int n_kv = (sc.Nk + kBN - 1) / kBN;
  it.nt0 = min(it.r0 / kBN + 1, n_kv);
  it.nt1 = min(it.r0 / kBN + 2, n_kv);
  it.lo0 = max(0, it.r0 - sc.window + 1) / kBN;
  it.lo1 = max(0, it.r0 + kBM - sc.window + 1) / kBN;
  return true;
}

__device__ __forceinline__ bool aborted(const WinBars* bars) {
  return *reinterpret_cast<const volatile int*>(&bars->abort) != 0;
}

template <Dt DT, bool ALIBI>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_window_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                          float* __restrict__ lse,
                          int Hq, int Hkv, int Nq, float sl2, const float* __restrict__ alibi, unsigned* status,
                          const WinSched sc) {
  constexpr int S = kWStages;
  constexpr bool kBF16 = DT == Dt::BF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;  // query tile t, buffer qb at sQ + (2 t + qb) * kWQBytes
  uint8_t* sK = sQ + 4 * kWQBytes;
  uint8_t* sV = sK + S * kWKVBytes;
  uint8_t* sO = sV + S * kWKVBytes;  // O staging of softmax warp w at sO + (w - 4) * 4 KB (1 KB aligned)
  WinBars* bars = reinterpret_cast<WinBars*>(sO + kWOStage);
  WinItem* items =
      reinterpret_cast<WinItem*>(reinterpret_cast<uint8_t*>(bars) + ((sizeof(WinBars) + 15) & ~size_t(15)));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t)
      for (int qb = 0; qb < 2; ++qb) {
        mbar_init(&bars->q_full[t][qb], 1);
        mbar_init(&bars->q_empty[t][qb], 1);
      }
    for (int i = 0; i < S; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 4 * 32);
      mbar_init(&bars->p_ready[t], 4 * 32);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_final[t], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  for (int x = threadIdx.x; x < kMaxItems; x += kThreads) {
    WinItem it;
    if (!win_item(sc, x, it)) it.bh = -1;
    items[x] = it;
  }
  if (warp == 1) {
    tc_alloc(&bars->tmem_base, kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * 168, "register split exceeds the launch budget");
  if (warp < 4) {
    regs_dec<kRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (whole warp, one lane issues)
      // Per item: its two query tiles into the item's Q buffer, then its key
      // tiles [lo0, nt1) through the K and V rings, whose slots are numbered
      // across items.
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int nk = 0, nv = 0;  // K and V tiles issued (all items)
      int kq = 0;          // items whose query tiles were issued; item k uses Q buffer k & 1
      bool ok = true;
      for (int k = 0; ok && k < kMaxItems; ++k) {
        const WinItem it = items[k];
        if (it.bh < 0 || aborted(bars)) break;
        const int qb = k & 1;
        const int kv_plane = (it.bh / Hq) * Hkv + (it.bh % Hq) / (Hq / Hkv);
        if (lane == 0)
          (void)RF_INB(it.bh < sc.BH && it.r0 < Nq && it.lo0 >= 0 && it.nt1 * kBN < sc.Nk + kBN &&
                           kv_plane < (sc.BH / Hq) * Hkv, status);
        if (k >= 2 && !(ok = mbar_wait_warp(&bars->q_empty[0][qb], ((k >> 1) - 1) & 1) &&
                             mbar_wait_warp(&bars->q_empty[1][qb], ((k >> 1) - 1) & 1)))
          break;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          mbar_expect_tx_elect(&bars->q_full[t][qb], kWQBytes);
          tma_load_3d_elect(sQ + (2 * t + qb) * kWQBytes, &tq, &bars->q_full[t][qb], 0, it.r0 + t * kBM, it.bh);
        }
        kq = k + 1;
        for (int j = it.lo0; ok && j < it.nt1; ++j) {
          const int key0 = j * kBN;
          int st = nk % S;
          if (nk >= S && !(ok = mbar_wait_warp(&bars->k_empty[st], ((nk / S) - 1) & 1))) break;
          mbar_expect_tx_elect(&bars->k_full[st], kWKVBytes);
          tma_load_3d_elect(sK + st * kWKVBytes, &tk, &bars->k_full[st], 0, key0, kv_plane);
          ++nk;
          st = nv % S;
          if (nv >= S && !(ok = mbar_wait_warp(&bars->v_empty[st], ((nv / S) - 1) & 1))) break;
          mbar_expect_tx_elect(&bars->v_full[st], kWKVBytes);
          tma_load_3d_elect(sV + st * kWKVBytes, &tv, &bars->v_full[st], 0, key0, kv_plane);
          ++nv;
        }
      }
      if (!ok) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        bars->abort = 1;
      }
      // every copy issued must land before the CTA exits
      bool drained = true;
      for (int k = kq > 2 ? kq - 2 : 0; k < kq; ++k)
        for (int t = 0; t < 2; ++t) drained &= mbar_wait_warp(&bars->q_full[t][k & 1], (k >> 1) & 1);
      for (int j = nk > S ? nk - S : 0; j < nk; ++j) drained &= mbar_wait_warp(&bars->k_full[j % S], (j / S) & 1);
      for (int j = nv > S ? nv - S : 0; j < nv; ++j) drained &= mbar_wait_warp(&bars->v_full[j % S], (j / S) & 1);
      if (!drained && lane == 0) atomicOr(status, kStatusTimeout);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (whole warp, one lane issues)
      // Per item: S of its first key tile, then one step per key tile j that
      // issues S_t of the next key tile (of this item or, at its last tile, of
      // the next item) for the query tiles that see it, and PV_t of tile j.
      // Barrier phases run on across items through the counts of S and PV
      // issued per query tile.
      constexpr uint32_t idS = tc_idesc_f16(kBF16, kBM, kBN, false);
      constexpr uint32_t idPV = tc_idesc_f16(kBF16, kBM, kWD, true);
      const uint64_t dQ = tc_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = tc_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = tc_sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      auto issue_s = [&](int t, int qb, int st) {  // S_t = Q_t K^T from Q buffer qb, K stage st
        const uint64_t a0 = dQ + static_cast<uint64_t>((2 * t + qb) * (kWQBytes >> 4));
        const uint64_t b0 = dK + static_cast<uint64_t>(st * (kWKVBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk)
          tc_mma_ss_elect(tmem + t * kBN, a0 + kk * 2, b0 + kk * 2, idS, kk > 0 ? 1u : 0u);
      };
      auto issue_pv = [&](int t, int st, bool acc) {  // O_t += P_t V from V stage st
        const uint64_t b0 = dV + static_cast<uint64_t>(st * (kWKVBytes >> 4));
        const uint32_t pcol = tmem + kWPCol + t * (kBN / 2);
        const uint32_t dO = tmem + kWOCol + t * kWD;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc_mma_ts_elect(dO, pcol + kk * 8, b0 + kk * (16 * 128 / 16), idPV, (acc || kk > 0) ? 1u : 0u);
      };
      WinItem it = items[0];  // the grid never exceeds the item count
      int lo0 = it.lo0, nt0 = it.nt0, lo1 = it.lo1, nt1 = it.nt1, k = 0;  // current item and its key tiles
      int ns0 = 0, ns1 = 0, np0 = 0, np1 = 0;  // S and PV issued per query tile (all items)
      bool ok = mbar_wait_warp(&bars->q_full[0][0], 0) && mbar_wait_warp(&bars->q_full[1][0], 0) &&
                mbar_wait_warp(&bars->k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0, 0);
        tc_commit_elect(&bars->s_full[0]);
        ns0 = 1;
        if (lo1 == lo0) {
          issue_s(1, 0, 0);
          tc_commit_elect(&bars->s_full[1]);
          ns1 = 1;
        }
        tc_commit_elect(&bars->k_empty[0]);
      }
      // The softmax of tile t reads O_t in an item's epilogue before it marks the
      // next item's first P_t ready, so p_ready also orders that item's first
      // PV_t (which overwrites O_t) after the read.
      int j = lo0, st = 0, ph = 0;  // current key tile, its ring stage and phase
      while (ok) {
        const int qb = k & 1;
        const bool last = j + 1 == nt1;  // the next key tile is the first of item k + 1
        WinItem nx;
        bool next = true, n_in0 = j + 1 < nt0, n_in1 = j + 1 >= lo1;
        int qbn = qb;
        if (last) {
          next = k + 1 < kMaxItems && !aborted(bars);
          if (next) {
            nx = items[k + 1];
            next = nx.bh >= 0;
          }
          qbn = (k + 1) & 1;
          if (next && !(ok = mbar_wait_warp(&bars->q_full[0][qbn], ((k + 1) >> 1) & 1) &&
                             mbar_wait_warp(&bars->q_full[1][qbn], ((k + 1) >> 1) & 1)))
            break;
          n_in0 = next;
          n_in1 = next && nx.lo1 == nx.lo0;
        }
        const int stn = st + 1 == S ? 0 : st + 1, phn = st + 1 == S ? ph ^ 1 : ph;  // stage / phase of the next tile
        bool k_ready = false;
        // S_t(next) as soon as softmax t has read S_t(current); PV_t(current) once P_t is ready.
        if (n_in0) {
          if (ns0 > 0 && !(ok = mbar_wait_warp(&bars->s_free[0], (ns0 - 1) & 1))) break;
          if (!(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
          k_ready = true;
          tc_fence_after();
          issue_s(0, qbn, stn);
          tc_commit_elect(&bars->s_full[0]);
          ++ns0;
        }
        if (!(ok = mbar_wait_warp(&bars->v_full[st], ph))) break;
        if (j < nt0) {
          if (!(ok = mbar_wait_warp(&bars->p_ready[0], np0 & 1))) break;
          tc_fence_after();
          issue_pv(0, st, j > lo0);
          tc_commit_elect(&bars->pv_done[0]);
          if (j == nt0 - 1) tc_commit_elect(&bars->o_final[0]);
          ++np0;
        }
        if (n_in1) {
          if (ns1 > 0 && !(ok = mbar_wait_warp(&bars->s_free[1], (ns1 - 1) & 1))) break;
          if (!k_ready && !(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
          tc_fence_after();
          issue_s(1, qbn, stn);
          tc_commit_elect(&bars->s_full[1]);
          ++ns1;
        }
        if (next) tc_commit_elect(&bars->k_empty[stn]);
        if (j >= lo1) {
          if (!(ok = mbar_wait_warp(&bars->p_ready[1], np1 & 1))) break;
          tc_fence_after();
          issue_pv(1, st, j > lo1);
          tc_commit_elect(&bars->pv_done[1]);
          if (j == nt1 - 1) tc_commit_elect(&bars->o_final[1]);
          ++np1;
        }
        tc_commit_elect(&bars->v_empty[st]);
        st = stn;
        ph = phn;
        if (!last) {
          ++j;
          continue;
        }
        // every S of item k has been issued: its Q buffer may be reloaded once they complete
        tc_commit_elect(&bars->q_empty[0][qb]);
        tc_commit_elect(&bars->q_empty[1][qb]);
        if (!next) break;
        ++k;
        j = nx.lo0;
        lo0 = nx.lo0;
        nt0 = nx.nt0;
        lo1 = nx.lo1;
        nt1 = nx.nt1;
      }
      if (!ok) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        bars->abort = 1;
      }
      // every MMA issued must complete before TMEM is released
      tc_commit_elect(&bars->drain);
      if (!mbar_wait_warp(&bars->drain, 0) && lane == 0) atomicOr(status, kStatusTimeout);
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax (one thread per query row)
    const int t = (warp - 4) >> 2;
    const int qw = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * kBN;
    const uint32_t tP = tmem + lane_off + kWPCol + t * (kBN / 2);
    const uint32_t tO = tmem + lane_off + kWOCol + t * kWD;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    int cnt = 0;   // key tiles this query tile has processed (all items): barrier phases
    int nfin = 0;  // items whose O this query tile has finished
    bool ok = true;
    for (int k = 0; ok && k < kMaxItems; ++k) {
      int row, jlo, jhi, bh;
      {
        const WinItem it = items[k];
        if (it.bh < 0 || aborted(bars)) break;
        bh = it.bh;
        row = it.r0 + t * kBM + qw * 32 + lane;
        jlo = t == 0 ? it.lo0 : it.lo1;
        jhi = t == 0 ? it.nt0 : it.nt1;
      }
      const float slope2 = ALIBI ? __ldg(alibi + (bh % Hq)) * kLog2e : 0.f;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = jlo; j < jhi; ++j, ++cnt) {
        const int jt = j - jlo;  // key tiles of this item so far
        if (!(ok = warp_wait(&bars->s_full[t], cnt & 1))) break;
        tc_fence_after();
        uint32_t s[kBN];
        tc_ld128(tS, s);  // the row's 128 scores in one load
        tc_wait_ld();
        tc_fence_before();  // S_t may be overwritten by the next S_t now
        mbar_arrive(&bars->s_free[t]);
        const int key0 = j * kBN;
        // columns below cl and from cf on are visible; a tile is cut by at most
        // the diagonal (or Nk) from above and the window's edge from below, and
        // each bound costs one compare per column only where some row needs it
        const int cl = min(sc.Nk, row + 1) - key0;
        const int cf = row - sc.window + 1 - key0;
        if (__any_sync(0xffffffffu, cl < kBN)) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= cl) s[c] = __float_as_uint(-INFINITY);
        }
        if (__any_sync(0xffffffffu, cf > 0)) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c < cf) s[c] = __float_as_uint(-INFINITY);
        }
        if constexpr (ALIBI) {
          // s <- s * scale * log2 e + slope * log2 e * (key - row), one packed FMA per
          // pair, the bias of pair e carried in packed accumulator e mod 4
          const float base = slope2 * static_cast<float>(key0 - row);
          uint64_t bias[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bias[q] = f2pack(fmaf(slope2, static_cast<float>(2 * q), base),
                             fmaf(slope2, static_cast<float>(2 * q + 1), base));
          const uint64_t step = f2pack(8.f * slope2, 8.f * slope2);
#pragma unroll
          for (int e = 0; e < kBN / 2; ++e) {
            const uint64_t r = fma_f32x2(u2pack(s[2 * e], s[2 * e + 1]), sl2x2, bias[e & 3]);
            f2unpack_u(r, s[2 * e], s[2 * e + 1]);
            bias[e & 3] = add_f32x2(bias[e & 3], step);
          }
        }
        // level 1: the tile max decides m; level 2: P = 2^(s*sl2 - m), all
        // exponentials before any wait below
        const float mt = scaled_max_from<0, ALIBI>(s, sl2);
        const bool need = mt > m_run + kRescaleThreshold;
        const float m_new = need ? mt : m_run;
        // a row can see no key of this tile: keep it at zero weight
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2_ftz(m_run - m_use);
        uint32_t pk[kBN / 2];
        const float tsum = exp_pairs<DT, ALIBI, 0, kBN / 2>(s, sl2x2, f2pack(-m_use, -m_use), pk);
        if (jt > 0) {  // the previous PV_t must be done before P_t and O_t are touched
          if (!(ok = warp_wait(&bars->pv_done[t], (cnt - 1) & 1))) break;
          tc_fence_after();
        }
        tc_st64(tP, pk);  // P of the row in one store
        l_run = fmaf(l_run, alpha, tsum);
        // level 3 correction: rescale O in TMEM when some row's max moved
        if (jt > 0 && __any_sync(0xffffffffu, need)) {
          const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
          for (int i = 0; i < kWD / 32; ++i) {
            uint32_t ov[32];
            tc_ld32(tO + 32 * i, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t r = mul_f32x2(u2pack(ov[e], ov[e + 1]), a2);
              f2unpack_u(r, ov[e], ov[e + 1]);
            }
            tc_st32(tO + 32 * i, ov);
          }
        }
        m_run = m_new;
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_ready[t]);
      }
      if (!ok) break;
      // no key tile for this query tile (all its rows past Nq): nothing to write
      if (jhi <= jlo) continue;
      if (!(ok = warp_wait(&bars->o_final[t], nfin & 1))) break;
      ++nfin;
      // epilogue: O / l in the output dtype, LSE in natural log.  The warp's 32
      // rows (4 KB, contiguous in O) go through its staging buffer in the
      // 128-byte swizzle of the O tensor map, and one TMA store writes them
      // (rows past Nq are clipped): a per-thread store of each 128-byte row
      // touched 32 lines per instruction.
      tc_fence_after();
      const float inv = 1.0f / l_run;
      const bool row_ok = row < Nq;
      const bool in_o = RF_INB(bh < sc.BH && row >= 0, status);
      uint8_t* ob = sO + (warp - 4) * (32 * kWD * 2);
      if (lane == 0) tma_store_wait_read();  // the previous item's store has read the buffer
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kWD / 32; ++i) {
        uint32_t ov[32];
        tc_ld32(tO + 32 * i, ov);
        tc_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = Pack<DT>::pack2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)  // 16-byte chunk 4 i + v4 of row `lane`, at chunk (4 i + v4) ^ (lane mod 8)
          *reinterpret_cast<uint4*>(ob + lane * 128 + ((((4 * i + v4) ^ lane) & 7) << 4)) =
              make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      }
      fence_proxy_async_smem();  // the staged rows are visible to the TMA store
      __syncwarp();
      const int wrow = row - lane;  // the warp's first row
      if (lane == 0 && wrow < Nq && in_o) {
        tma_store_3d(&to, ob, 0, wrow, bh);
        tma_store_commit();
      }
      if (row_ok && in_o && lse) lse[static_cast<long long>(bh) * Nq + row] = (m_run + log2f(l_run)) * kLn2;
      // O_t has been read (tcgen05.ld waited); the fence before this thread's
      // next p_ready arrival lets the next item's first PV_t overwrite it
    }
    if (!ok) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      bars->abort = 1;
    }
    if (lane == 0) tma_store_wait_read();  // the staging buffer has been read before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
}

template <Dt DT, bool ALIBI>
cudaError_t launch_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, float scale, int window, const float* alibi, unsigned* status, int sms,
                          cudaStream_t s) {
  alignas(64) CUtensorMap tq, tk, tv, to;
  cudaError_t err = cudaSuccess;
  if (!encode_tma_3d_16bit(&tq, q, kWD, Nq, uint64_t(B) * Hq, kBM, &err)) return err;
  if (!encode_tma_3d_16bit(&to, o, kWD, Nq, uint64_t(B) * Hq, 32, &err)) return err;  // one warp's rows
  if (!encode_tma_3d_16bit(&tk, k, kWD, Nk, uint64_t(B) * Hkv, kBN, &err)) return err;
  if (!encode_tma_3d_16bit(&tv, v, kWD, Nk, uint64_t(B) * Hkv, kBN, &err)) return err;
  const int nqt = (Nq + 2 * kBM - 1) / (2 * kBM);
  const long long n_items = static_cast<long long>(nqt) * B * Hq;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  WinSched sc;
  sc.BH = B * Hq;
  sc.nqt = nqt;
  sc.Nk = Nk;
  sc.window = window;
  sc.n_items = static_cast<int>(n_items);
  // one CTA per SM (at most kMaxItems items each); without an SM count, one per item
  long long ctas = sms > 0 && sms < n_items ? sms : n_items;
  const long long min_ctas = (n_items + kMaxItems - 1) / kMaxItems;
  if (ctas < min_ctas) ctas = min_ctas;
  const int smem = kWTiles + kWOStage + 1024 + static_cast<int>((sizeof(WinBars) + 15) & ~size_t(15)) +
                   kMaxItems * static_cast<int>(sizeof(WinItem)) + 64;
  auto kern = attn_tc_window_kernel<DT, ALIBI>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<static_cast<unsigned>(ctas), kThreads, smem, s>>>(tq, tk, tv, to, lse, Hq, Hkv, Nq,
                                                           scale * kLog2e, alibi, status, sc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Nq, int Nk, float scale, int window, const float* alibi, Dt dt,
                                  unsigned* status, int sms, cudaStream_t s) {
#define RF_WIN_ARGS q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, window, alibi, status, sms, s
  if (dt == Dt::BF16)
    return alibi ? launch_window<Dt::BF16, true>(RF_WIN_ARGS) : launch_window<Dt::BF16, false>(RF_WIN_ARGS);
  if (dt == Dt::F16)
    return alibi ? launch_window<Dt::F16, true>(RF_WIN_ARGS) : launch_window<Dt::F16, false>(RF_WIN_ARGS);
#undef RF_WIN_ARGS
  return cudaErrorNotSupported;
}

}  // namespace rf
