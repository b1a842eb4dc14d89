// attn_fwd_tc.cuh -- attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for fp16/bf16 inputs, D in {64, 128}: the kernel
// template and its launchers, instantiated without rotary embedding in
// attn_fwd_tc.cu and with it in attn_fwd_tc_rope.cu (two translation units
// that compile in parallel).
//
// The cascade max -> sum exp -> sum exp*v (RedFuser, Abstract: safe softmax
// followed by GEMM; "Operator Fusion" guide, section 2, Pattern 4) runs as one
// loop over 128-key tiles in the incremental form of RedFuser's Figure 4:
// level 1 (reduce max, combine +) keeps a running row max m; levels 2 and 3
// (reduce +, combine *) keep the running sum l and the running output O, both
// corrected by exp(m_old - m_new) when m rises.  The correction is applied
// lazily, which stays exact because l and O are always built against the same
// m: m moves only when a tile's max exceeds it by more than 2^8 (in base 2),
// which keeps P <= 256.  Non-causal D = 64 rows speculate: once m is finite, P
// is formed against it without scanning the tile, and m moves only when a half
// row's sum of P exceeds 2^15, so P stays <= 2^15.
//
// CTA = two query tiles of 128 rows (rows r0..r0+255 of one (batch, head)),
// 12 warps:
//   warp 0      TMA producer: Q once; K and V tiles through 2-3 stage rings
//               (at D = 64 a stage's K and V share one full/empty barrier
//               pair, freed once PV_1 of the tile is done: one wait and one
//               commit fewer per tile on the MMA warp).
//   warp 1      allocates 512 TMEM columns and issues every tcgen05.mma.
// Both run their loops as a whole warp with warp-uniform operands; one lane
// issues through an elect.sync predicate (no divergent branch), which keeps
// the issue cost at the tensor core's own rate.
//   warps 4-7   softmax for query tile 0, warps 8-11 for tile 1: one thread
//               per query row, i.e. per TMEM lane, so row max and row sum need
//               no cross-thread reduction.
// Registers are re-split after launch: warps 0-3 drop to 80 per thread and
// the softmax warps rise to 208 (a row of S is 128 registers).
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
//  * D = 64: P0 [384,448) and P1 [448,512) have columns of their own (16-bit,
//    two per column).  Softmax frees S_t as soon as it has loaded it, so the
//    MMA issuer runs S_t(j+1) while softmax still exponentiates tile j; PV_t(j)
//    follows once P_t(j) is ready.  Softmax waits for PV_t(j-1) to complete
//    before it overwrites P_t or rescales O_t.
//  * D = 128: no spare columns; P_t overwrites the first 64 columns of S_t and
//    the order per key tile is PV0_j, S0_{j+1}, PV1_j, S1_{j+1}, so the tensor
//    core works on one tile while the other tile's softmax runs (ping-pong).
//    A commit after S_t(j+1) then also covers PV_t(j).
// In both cases P is the TMEM A operand of O += P V.
//
// Shared memory operands use the 128-byte swizzle written by TMA: Q and K
// K-major (boxes of 64 dims x 128 rows), V MN-major (the same boxes read as
// D x keys).  Causal CTAs are scheduled longest-first, and the query heads of
// one GQA group are adjacent in launch order so their K/V tiles hit in L2.
//
// Split tail (no mask, caller workspace given): with one CTA per SM, U units
// of 256 query rows take ceil(U / SMs) waves, and a last wave of a few units
// leaves most SMs idle for a whole unit.  The last U mod SMs units are then
// split along the keys into n_split pieces each (one CTA per piece), which
// write their normalised partial O_s and lse_s in fp32 to the workspace; the
// log-sum-exp merge (RedFuser, Figure 13: the FlashDecoding split and merge)
// then writes those rows of O and LSE.
// Causal sliding windows of up to kWindowPersistMax keys at D = 64 go to the
// persistent kernel of attn_fwd_tc_window.cu instead: their units are too short
// to amortise a CTA each.
// Rotary embedding at the load (ROPE >= 1): AttnFuse (Figure 1, Table 4)
// fuses the rotation of Q and K into its attention kernel.  Here each softmax
// thread turns its own Q row in shared memory once, right after TMA lands it
// and before the first S; with ROPE = 2 two otherwise idle warps (2 and 3)
// also turn the K rows of every ring stage before S reads them, which every
// CTA streaming that tile repeats.  The angles come from rope_angle.cuh, the
// same function the separate pass (rope.cu) uses.
// Every mbarrier wait is bounded; on a timeout the CTA records RF_ERR_TIMEOUT,
// waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <math.h>

#include "attn_tc_common.cuh"
#include "lse_merge.cuh"
#include "rf_device.cuh"
#include "rope_angle.cuh"

namespace rf {
namespace {

// Speculative P (rows with a finite running max): every P of a half row stays
// <= 2^kSpecLog2, far inside fp16's range, or the half is redone.
constexpr float kSpecLog2 = 15.0f;
constexpr float kSpecMax = 32768.0f;  // 2^kSpecLog2

template <int D>
struct Cfg {
  static constexpr int kQBytes = kBM * D * 2;    // one query tile
  static constexpr int kKVBytes = kBN * D * 2;   // one K or V tile
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kTiles = 2 * kQBytes + 2 * kStages * kKVBytes;
  static constexpr bool kSepP = D == 64;         // P in columns of its own
  static constexpr int kOCol = 2 * kBN;          // O0 at 256, O1 at 256 + D
  static constexpr int kPCol = 2 * kBN + 2 * D;  // P0 at 384, P1 at 448 (D = 64)
  // K rotation tables (rotary embedding of K inside the kernel): (cos, sin) of
  // b * theta_i for b < 32, laid out [i][b], and of the tile's base positions
  // key0 + 32 a for a < 4, laid out [a][i].
  static constexpr int kRopeR = 32 * (D / 2);
  static constexpr int kRopeB = (kBN / 32) * (D / 2);
  static constexpr int kRopeBytes = (kRopeR + kRopeB) * 8;
};

struct alignas(8) TcBars {
  uint64_t q_full, q_rot, k_rot[3], rope_tab;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], s_free[2], p_ready[2], pv_done[2], o_final[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Output rows of the split tail's partial rows (partial row g = row g % 256 of
// tail unit g / 256); rows past Nq are skipped.
struct AttnTailRows {
  int first_unit, BH, nqt, Nq;
  __device__ __forceinline__ long long operator()(long long g) const {
    int c, bh;
    unit_coords(first_unit + static_cast<int>(g / (2 * kBM)), BH, nqt, c, bh);
    const int q = c * 2 * kBM + static_cast<int>(g % (2 * kBM));
    return q < Nq ? static_cast<long long>(bh) * Nq + q : -1;
  }
};

// MASK: 0 none, 1 causal (top-left), 2 causal with a sliding window of
// `window` keys (key j visible to query i iff i - window < j <= i).
// ALIBI: add slope_h * (j - i) to each scaled score (slopes per query head).
// ROPE: 0 none; 1 rotate the Q rows (rotary embedding at position
// rope_pos + row) in shared memory after their load; 2 also the K rows of
// every key tile (at rope_pos + key) before S reads them.
template <Dt DT, int D, int MASK, bool ALIBI, int ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                   float* __restrict__ lse,
                   int Hq, int Hkv, int Nq, int Nk, int BH, int nqt, float sl2, int window,
                   const float* __restrict__ alibi, unsigned* status, int n_full, int n_split,
                   float* __restrict__ o_part, float* __restrict__ lse_part,
                   const __grid_constant__ RopeParams rope, int rope_pos, int batch_major, int prefetch_stride) {
  constexpr bool CAUSAL = MASK >= 1;
  constexpr bool kSpec = D == 64 && MASK == 0 && !ALIBI;
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  static_assert(C::kOCol + 2 * D <= kTmemCols && (!C::kSepP || C::kPCol + kBN <= kTmemCols),
                "TMEM columns of S, O and P must fit the allocation");
  constexpr bool kBF16 = DT == Dt::BF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + 2 * C::kQBytes;
  uint8_t* sV = sK + S * C::kKVBytes;
  float2* sRopeR = reinterpret_cast<float2*>(sV + S * C::kKVBytes);  // only with ROPE == 2
  float2* sRopeB = sRopeR + C::kRopeR;
  TcBars* bars = reinterpret_cast<TcBars*>(sV + S * C::kKVBytes + (ROPE == 2 ? C::kRopeBytes : 0));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTAs from n_full on are pieces of the split tail: piece p is key range
  // p % n_split of unit n_full + p / n_split.
  const int id = blockIdx.x;
  const bool piece = MASK == 0 && id >= n_full;
  const int unit = piece ? n_full + (id - n_full) / n_split : id;
  const int split = piece ? (id - n_full) % n_split : 0;
  // unit -> query-tile pair c and batch*head bh
  auto coords = [&](int u, int& cc, int& bhh) {
    if (CAUSAL && batch_major) {
      // Batch-major order (longest units first within each batch): only one
      // batch's K and V tiles are live in L2 at a time, for when every head's K
      // and V together would not stay there.
      const int per_b = Hq * nqt;
      const int bb = u / per_b, r = u - bb * per_b;
      cc = nqt - 1 - r / Hq;
      bhh = bb * Hq + (r - (r / Hq) * Hq);
    } else {
      unit_coords(u, BH, nqt, cc, bhh);
    }
  };
  int c, bh;
  coords(unit, c, bh);
  const int h = bh % Hq, b = bh / Hq;
  const int kv_plane = b * Hkv + h / (Hq / Hkv);
  const int r0 = c * 2 * kBM;
  // Key tiles [lo_t, nt_t) that query tile t can see; the CTA streams
  // [lo0, nt1) (tile 1's rows come after tile 0's, so lo0 <= lo1, nt0 <= nt1).
  const int n_kv = (Nk + kBN - 1) / kBN;
  // a piece's key tiles: [floor(split n_kv / n_split), floor((split + 1) n_kv / n_split)), never empty
  const int plo = piece ? static_cast<int>(static_cast<long long>(split) * n_kv / n_split) : 0;
  const int phi = piece ? static_cast<int>(static_cast<long long>(split + 1) * n_kv / n_split) : n_kv;
  const int nt0 = CAUSAL ? min(r0 / kBN + 1, n_kv) : phi;
  const int nt1 = CAUSAL ? min(r0 / kBN + 2, n_kv) : phi;
  const int lo0 = MASK == 2 ? max(0, r0 - window + 1) / kBN : plo;
  const int lo1 = MASK == 2 ? max(0, r0 + kBM - window + 1) / kBN : plo;
  const int n_load = nt1 - lo0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_rot, 8 * 32);  // every softmax thread rotates its own row
    mbar_init(&bars->rope_tab, 2 * 32);
    for (int i = 0; i < S; ++i) {
      mbar_init(&bars->k_rot[i], 2 * 32);  // the two K-rotating warps
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
  // The producer warp (whose lane 0 initialised the barriers) starts the copies
  // that need no wait, Q and the first ring stages, before the CTA-wide barrier:
  // they overlap the TMEM allocation and the barrier itself.
  const int n_early = min(S, n_load);
  if (warp == 0) {
    __syncwarp();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    if (lane == 0) (void)RF_INB(bh < BH && r0 < Nq && kv_plane < (BH / Hq) * Hkv && lo0 >= 0 && nt1 <= n_kv, status);
    mbar_expect_tx_elect(&bars->q_full, 2 * C::kQBytes);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
        tma_load_3d_elect(sQ + t * C::kQBytes + bx * (kBM * 128), &tq, &bars->q_full, bx * 64, r0 + t * kBM, bh);
    // With one CTA per SM, CTA id + prefetch_stride is about the one that takes
    // this SM (or another) next: its Q tiles go to L2 now, so that its own
    // first load, which nothing overlaps, does not wait on HBM.  Only at
    // D = 128 (64 KB of Q per unit): there it saves 0.6%; at D = 64 it saved
    // nothing and part of the prefetched Q was evicted before use (DRAM reads
    // 88 -> 104 MB at B=4 H=12 N=4096).
    const int nid = id + prefetch_stride;
    if (prefetch_stride > 0 && nid < static_cast<int>(gridDim.x)) {
      const int nunit = MASK == 0 && nid >= n_full ? n_full + (nid - n_full) / n_split : nid;
      int nc, nbh;
      coords(nunit, nc, nbh);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) tma_prefetch_l2_3d_elect(&tq, bx * 64, nc * 2 * kBM + t * kBM, nbh);
    }
    for (int jj = 0; jj < n_early; ++jj) {  // ring slot jj holds key tile lo0 + jj
      const int key0 = (lo0 + jj) * kBN;
      if (lane == 0) (void)RF_INB(key0 < Nk, status);
      mbar_expect_tx_elect(&bars->k_full[jj], C::kSepP ? 2 * C::kKVBytes : C::kKVBytes);
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
        tma_load_3d_elect(sK + jj * C::kKVBytes + bx * (kBN * 128), &tk, &bars->k_full[jj], bx * 64, key0, kv_plane);
      uint64_t* vbar = C::kSepP ? &bars->k_full[jj] : &bars->v_full[jj];  // V rides on K's barrier at D = 64
      if (!C::kSepP) mbar_expect_tx_elect(vbar, C::kKVBytes);
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
        tma_load_3d_elect(sV + jj * C::kKVBytes + bx * (kBN * 128), &tv, vbar, bx * 64, key0, kv_plane);
    }
  }
  if (warp == 1) {
    tc_alloc(&bars->tmem_base, kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // The merge of a split tail (if any) may be scheduled once every CTA has
  // started; it waits on the device for this grid to complete.
  griddep_launch_dependents();

  // Register split: 128 x 80 (producer / MMA warpgroup) + 256 x 208 (softmax)
  // = 63,488 <= 384 x 168 registers granted at launch.
  static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * 168, "register split exceeds the launch budget");
  if (warp < 4) {
    regs_dec<kRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (whole warp, one lane issues)
      // Q and key tiles [0, n_early) were issued before the CTA-wide barrier.
      int issued_k = n_early, issued_v = C::kSepP ? 0 : n_early;
      bool ok = true;
      for (int jj = n_early; jj < n_load; ++jj) {  // ring slot jj % S holds key tile lo0 + jj
        const int st = jj % S, key0 = (lo0 + jj) * kBN;
        if (lane == 0) (void)RF_INB(key0 < Nk, status);
        if (jj >= S && !(ok = mbar_wait_warp(&bars->k_empty[st], ((jj / S) - 1) & 1))) break;
        mbar_expect_tx_elect(&bars->k_full[st], C::kSepP ? 2 * C::kKVBytes : C::kKVBytes);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_3d_elect(sK + st * C::kKVBytes + bx * (kBN * 128), &tk, &bars->k_full[st], bx * 64, key0, kv_plane);
        ++issued_k;
        if constexpr (C::kSepP) {  // V rides on K's barriers: one wait and one commit per stage
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx)
            tma_load_3d_elect(sV + st * C::kKVBytes + bx * (kBN * 128), &tv, &bars->k_full[st], bx * 64, key0, kv_plane);
          continue;
        }
        if (jj >= S && !(ok = mbar_wait_warp(&bars->v_empty[st], ((jj / S) - 1) & 1))) break;
        mbar_expect_tx_elect(&bars->v_full[st], C::kKVBytes);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_3d_elect(sV + st * C::kKVBytes + bx * (kBN * 128), &tv, &bars->v_full[st], bx * 64, key0, kv_plane);
        ++issued_v;
      }
      if (!ok) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        bars->abort = 1;
      }
      // every copy issued must land before the CTA exits
      bool drained = mbar_wait_warp(&bars->q_full, 0);
      for (int j = issued_k > S ? issued_k - S : 0; j < issued_k; ++j)
        drained &= mbar_wait_warp(&bars->k_full[j % S], (j / S) & 1);
      for (int j = issued_v > S ? issued_v - S : 0; j < issued_v; ++j)
        drained &= mbar_wait_warp(&bars->v_full[j % S], (j / S) & 1);
      if (!drained && lane == 0) atomicOr(status, kStatusTimeout);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (whole warp, one lane issues)
      // Issue cost matters here (one lane issues every MMA), so the whole warp
      // runs this loop with warp-uniform operands and elect.sync predicates the
      // instructions; the shared memory descriptors are built once: a K-step or
      // a ring stage only moves the 14-bit start-address field.
      constexpr uint32_t idS = tc_idesc_f16(kBF16, kBM, kBN, false);
      constexpr uint32_t idPV = tc_idesc_f16(kBF16, kBM, D, true);
      const uint64_t dQ = tc_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = tc_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = tc_sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      auto issue_s = [&](int t, int st) {  // S_t = Q_t K^T from K stage st  (M=128, N=128, K=D)
        const uint64_t a0 = dQ + static_cast<uint64_t>(t * (C::kQBytes >> 4));
        const uint64_t b0 = dK + static_cast<uint64_t>(st * (C::kKVBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr int kStepQ = kBM * 128 / 16, kStepK = kBN * 128 / 16;  // one 64-dim box
          const uint32_t oq = (kk >> 2) * kStepQ + (kk & 3) * 2, ok_ = (kk >> 2) * kStepK + (kk & 3) * 2;
          tc_mma_ss_elect(tmem + t * kBN, a0 + oq, b0 + ok_, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int st, bool acc) {  // O_t += P_t V from V stage st  (M=128, N=D, K=128)
        const uint64_t b0 = dV + static_cast<uint64_t>(st * (C::kKVBytes >> 4));
        const uint32_t pcol = tmem + (C::kSepP ? C::kPCol + t * (kBN / 2) : t * kBN);
        const uint32_t dO = tmem + C::kOCol + t * D;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc_mma_ts_elect(dO, pcol + kk * 8, b0 + kk * (16 * 128 / 16), idPV, (acc || kk > 0) ? 1u : 0u);
      };
      // Key tile j (ring slot jj = j - lo0) feeds query tile t when lo_t <= j < nt_t;
      // barrier phases of tile t count its own key tiles (j - lo_t).
      auto in0 = [&](int j) { return j >= lo0 && j < nt0; };
      auto in1 = [&](int j) { return j >= lo1 && j < nt1; };
      bool ok = mbar_wait_warp(ROPE ? &bars->q_rot : &bars->q_full, 0) && mbar_wait_warp(&bars->k_full[0], 0) &&
                (ROPE != 2 || mbar_wait_warp(&bars->k_rot[0], 0));
      if (ok) {
        tc_fence_after();
        if (in0(lo0)) {
          issue_s(0, 0);
          tc_commit_elect(&bars->s_full[0]);
        }
        if (in1(lo0)) {
          issue_s(1, 0);
          tc_commit_elect(&bars->s_full[1]);
        }
        if constexpr (!C::kSepP) tc_commit_elect(&bars->k_empty[0]);
      }
      int st = 0, ph = 0;  // ring stage and phase of key tile j
      for (int jj = 0; ok && jj < n_load; ++jj) {
        const int j = lo0 + jj, jn = j + 1;
        const int stn = st + 1 == S ? 0 : st + 1, phn = st + 1 == S ? ph ^ 1 : ph;  // stage / phase of j+1
        bool k_ready = false;
        if constexpr (C::kSepP) {
          // S_t(j+1) as soon as softmax t has read S_t(j); PV_t(j) once P_t(j) is ready.
          if (in0(jn)) {
            if (jn > lo0 && !(ok = mbar_wait_warp(&bars->s_free[0], (jn - 1 - lo0) & 1))) break;
            if (!(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
            if (ROPE == 2 && !(ok = mbar_wait_warp(&bars->k_rot[stn], phn))) break;
            k_ready = true;
            tc_fence_after();
            issue_s(0, stn);
            tc_commit_elect(&bars->s_full[0]);
          }
          if (in0(j)) {
            if (!(ok = mbar_wait_warp(&bars->p_ready[0], (j - lo0) & 1))) break;
            tc_fence_after();
            issue_pv(0, st, j > lo0);
            tc_commit_elect(&bars->pv_done[0]);
            if (j == nt0 - 1) tc_commit_elect(&bars->o_final[0]);
          }
          if (in1(jn)) {
            if (jn > lo1 && !(ok = mbar_wait_warp(&bars->s_free[1], (jn - 1 - lo1) & 1))) break;
            if (!k_ready && !(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
            if (!k_ready && ROPE == 2 && !(ok = mbar_wait_warp(&bars->k_rot[stn], phn))) break;
            tc_fence_after();
            issue_s(1, stn);
            tc_commit_elect(&bars->s_full[1]);
          }
          if (in1(j)) {
            if (!(ok = mbar_wait_warp(&bars->p_ready[1], (j - lo1) & 1))) break;
            tc_fence_after();
            issue_pv(1, st, j > lo1);
            tc_commit_elect(&bars->pv_done[1]);
            if (j == nt1 - 1) tc_commit_elect(&bars->o_final[1]);
          }
          tc_commit_elect(&bars->k_empty[st]);  // K and V of tile j: both stages free once PV_1(j) is done
        } else {
          // P aliases S: PV_t(j) must be issued before S_t(j+1) overwrites it.
          if (!(ok = mbar_wait_warp(&bars->v_full[st], ph))) break;
          if (in0(j)) {
            if (!(ok = mbar_wait_warp(&bars->p_ready[0], (j - lo0) & 1))) break;
            tc_fence_after();
            issue_pv(0, st, j > lo0);
            if (j == nt0 - 1) tc_commit_elect(&bars->o_final[0]);
          }
          if (in0(jn)) {
            if (!(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
            if (ROPE == 2 && !(ok = mbar_wait_warp(&bars->k_rot[stn], phn))) break;
            k_ready = true;
            tc_fence_after();
            issue_s(0, stn);
            tc_commit_elect(&bars->s_full[0]);
          }
          if (in1(j)) {
            if (!(ok = mbar_wait_warp(&bars->p_ready[1], (j - lo1) & 1))) break;
            tc_fence_after();
            issue_pv(1, st, j > lo1);
            if (j == nt1 - 1) tc_commit_elect(&bars->o_final[1]);
          }
          tc_commit_elect(&bars->v_empty[st]);
          if (in1(jn)) {
            if (!k_ready) {
              if (!(ok = mbar_wait_warp(&bars->k_full[stn], phn))) break;
              if (ROPE == 2 && !(ok = mbar_wait_warp(&bars->k_rot[stn], phn))) break;
              tc_fence_after();
            }
            issue_s(1, stn);
            tc_commit_elect(&bars->s_full[1]);
          }
          if (jn < nt1) tc_commit_elect(&bars->k_empty[stn]);
        }
        st = stn;
        ph = phn;
      }
      if (!ok) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        bars->abort = 1;
      }
      // every MMA issued must complete before TMEM is released
      tc_commit_elect(&bars->drain);
      if (!mbar_wait_warp(&bars->drain, 0) && lane == 0) atomicOr(status, kStatusTimeout);
    } else if (ROPE == 2) {
      // ---------------------------------------------------------- K rotation (warps 2 and 3)
      // The rows of every key tile are turned in place once TMA has landed
      // them, before S reads them.  The angle of key r of the tile is
      // (key0 + 32 a + b) theta_i with r = 32 a + b, so its (cos, sin) is the
      // complex product of a per-tile base (key0 + 32 a) theta_i and b theta_i
      // from a table built once per CTA: a few sincos per lane per tile
      // instead of one per element.  Warp 2 turns rows 0-63 (a = 0, 1), warp 3
      // rows 64-127 (a = 2, 3); each keeps the bases of its own rows, so the
      // two warps meet only once, on an mbarrier, after building the table.
      constexpr int H2 = D / 2;
      const int w2 = warp - 2;
      for (int e = w2 * 32 + lane; e < C::kRopeR; e += 64) {
        const int i = e >> 5, b = e & 31;  // [i][b]: a warp's 32 rows read 32 consecutive entries
        sRopeR[e] = rope_cs(static_cast<float>(b), i, rope);
      }
      mbar_arrive(&bars->rope_tab);
      bool ok = mbar_wait_warp(&bars->rope_tab, 0);
      float2* base = sRopeB + w2 * 2 * H2;  // [h][i] for this warp's a = 2 w2 + h
      for (int jj = 0; ok && jj < n_load; ++jj) {
        const int st = jj % S, key0 = (lo0 + jj) * kBN;
        __syncwarp();  // the previous tile's bases are no longer read
        for (int e = lane; e < 2 * H2; e += 32) {
          const int h = e / H2, i = e - h * H2;
          base[e] = rope_cs(static_cast<float>(rope_pos + key0 + 32 * (2 * w2 + h)), i, rope);
        }
        __syncwarp();
        if (!(ok = mbar_wait_warp(&bars->k_full[st], (jj / S) & 1))) break;
        (void)RF_INB(st < S && w2 >= 0 && w2 < 2, status);
        uint8_t* tile = sK + st * C::kKVBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = 64 * w2 + 32 * h + lane;  // key row of the tile: a = 2 w2 + h, b = lane
          const float2* bh = base + h * H2;
          const float2* rtab = sRopeR + lane;
#pragma unroll
          for (int gc = 0; gc < D / 16; ++gc) {
            const int gb = gc + D / 16;  // the partner chunk: dims + D/2
            uint4* pa = reinterpret_cast<uint4*>(tile + (gc >> 3) * (kBN * 128) + r * 128 + (((gc & 7) ^ (r & 7)) << 4));
            uint4* pb = reinterpret_cast<uint4*>(tile + (gb >> 3) * (kBN * 128) + r * 128 + (((gb & 7) ^ (r & 7)) << 4));
            float xa[8], xb[8], ya[8], yb[8];
            Pack<DT>::unpack(*pa, xa);
            Pack<DT>::unpack(*pb, xb);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int i = gc * 8 + e;
              const float2 bc = bh[i], rc = rtab[i * 32];
              const float2 cs = make_float2(fmaf(bc.x, rc.x, -bc.y * rc.y), fmaf(bc.y, rc.x, bc.x * rc.y));
              rope_rotate(xa[e], xb[e], cs, ya[e], yb[e]);
            }
            *pa = Pack<DT>::pack(ya);
            *pb = Pack<DT>::pack(yb);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core's reads
        mbar_arrive(&bars->k_rot[st]);
      }
      if (!ok) {
        if (lane == 0) atomicOr(status, kStatusTimeout);
        bars->abort = 1;
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax (one thread per query row)
    const int t = (warp - 4) >> 2;
    const int qw = warp & 3;
    const int row = r0 + t * kBM + qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * kBN;
    const uint32_t tP = tmem + lane_off + (C::kSepP ? C::kPCol + t * (kBN / 2) : t * kBN);
    const uint32_t tO = tmem + lane_off + C::kOCol + t * D;
    const int jlo = t == 0 ? lo0 : lo1, jhi = t == 0 ? nt0 : nt1;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    const float slope2 = ALIBI ? __ldg(alibi + (bh % Hq)) * kLog2e : 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool spec = kSpec;  // warp-uniform: cleared by the first failed speculation
    bool ok = true;
    if constexpr (ROPE >= 1) {
      // Rotary embedding of this thread's own query row in shared memory, once,
      // before any S reads Q: the pair (i, i + D/2) at position rope_pos + row.
      ok = warp_wait(&bars->q_full, 0);
      if (ok) {
        const int rl = qw * 32 + lane;  // row within the tile
        (void)RF_INB(rl < kBM && t < 2, status);
        uint8_t* qrow = sQ + t * C::kQBytes + rl * 128;
        const float p = static_cast<float>(rope_pos + row);
#pragma unroll
        for (int gc = 0; gc < D / 16; ++gc) {
          const int gb = gc + D / 16;
          uint4* pa = reinterpret_cast<uint4*>(qrow + (gc >> 3) * (kBM * 128) + (((gc & 7) ^ (rl & 7)) << 4));
          uint4* pb = reinterpret_cast<uint4*>(qrow + (gb >> 3) * (kBM * 128) + (((gb & 7) ^ (rl & 7)) << 4));
          float xa[8], xb[8], ya[8], yb[8];
          Pack<DT>::unpack(*pa, xa);
          Pack<DT>::unpack(*pb, xb);
#pragma unroll
          for (int e = 0; e < 8; ++e) rope_rotate(xa[e], xb[e], rope_cs(p, gc * 8 + e, rope), ya[e], yb[e]);
          *pa = Pack<DT>::pack(ya);
          *pb = Pack<DT>::pack(yb);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core's reads
      }
      mbar_arrive(&bars->q_rot);
    }
    for (int j = jlo; ok && j < jhi; ++j) {
      const int jt = j - jlo;  // this tile's own key-tile count: barrier phases
      if (!(ok = warp_wait(&bars->s_full[t], jt & 1))) break;
      tc_fence_after();
      uint32_t s[kBN];
      tc_ld128(tS, s);  // the row's 128 scores in one load
      tc_wait_ld();
      if constexpr (C::kSepP) {  // S_t may be overwritten by S_t(j+1) now
        tc_fence_before();
        mbar_arrive(&bars->s_free[t]);
      }
      const int key0 = j * kBN;
      if constexpr (CAUSAL) {
        // columns below cl and from cf on are visible; each bound costs one
        // compare per column only where some row of the warp needs it
        const int cl = min(Nk, row + 1) - key0;
        if (__any_sync(0xffffffffu, cl < kBN)) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= cl) s[c] = __float_as_uint(-INFINITY);
        }
        if constexpr (MASK == 2) {
          const int cf = row - window + 1 - key0;
          if (__any_sync(0xffffffffu, cf > 0)) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c < cf) s[c] = __float_as_uint(-INFINITY);
          }
        }
      } else if (key0 + kBN > Nk) {
        const int lim = Nk, first = 0;  // keys below lim and from first on are visible
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c >= lim || key0 + c < first) s[c] = __float_as_uint(-INFINITY);
      }
      if constexpr (ALIBI) {
        // s <- s * scale * log2 e + slope * log2 e * (key - row), one packed FMA per
        // pair: the bias of the pair (2e, 2e+1) rides in one of four packed
        // accumulators that advance by 8 * slope per pair of their own.
        const float base = slope2 * static_cast<float>(key0 - row);
        uint64_t bias[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          bias[k] = f2pack(fmaf(slope2, static_cast<float>(2 * k), base),
                           fmaf(slope2, static_cast<float>(2 * k + 1), base));
        const uint64_t step = f2pack(8.f * slope2, 8.f * slope2);
#pragma unroll
        for (int e = 0; e < kBN / 2; ++e) {
          const uint64_t r = fma_f32x2(u2pack(s[2 * e], s[2 * e + 1]), sl2x2, bias[e & 3]);
          f2unpack_u(r, s[2 * e], s[2 * e + 1]);
          bias[e & 3] = add_f32x2(bias[e & 3], step);
        }
      }
      uint32_t pk[kBN / 2];
      float m_new = m_run, tsum = 0.f;
      bool need = false;
      // Speculation (non-causal D = 64 without ALiBi): a row whose running max m
      // is finite first forms P against m without scanning the tile, which is
      // exact as long as no P exceeds kSpecMax; the sum of each half row bounds
      // that.  When a first half fails, the row is redone from the tile max;
      // when only a second half fails, that half is rescanned alone.  After one
      // failure the warp stops speculating (steadily rising scores would make
      // it fail on every tile).
      if constexpr (kSpec) {
        bool exact = !spec || __any_sync(0xffffffffu, m_run == -INFINITY);
        float h0, h1;
        for (;;) {
          if (exact) {
            const float mt = scaled_max_from<0, ALIBI>(s, sl2);
            m_new = mt > m_run + kRescaleThreshold ? mt : m_run;
          }
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const uint64_t negm2 = f2pack(-m_use, -m_use);
          h0 = exp_pairs<DT, ALIBI, 0, kBN / 4>(s, sl2x2, negm2, pk);
          if (exact) {
            h1 = exp_pairs<DT, ALIBI, kBN / 4, kBN / 2>(s, sl2x2, negm2, pk);
            break;
          }
          if (!__any_sync(0xffffffffu, !(h0 <= kSpecMax))) {
            h1 = exp_pairs<DT, ALIBI, kBN / 4, kBN / 2>(s, sl2x2, negm2, pk);
            const bool big = !(h1 <= kSpecMax);
            if (__any_sync(0xffffffffu, big)) {
              // every first-half P is <= 2^kSpecLog2, so m + kSpecLog2 bounds that half
              spec = false;
              const float mt = scaled_max_from<kBN / 2, ALIBI>(s, sl2);
              m_new = big ? fmaxf(mt, m_run + kSpecLog2) : m_run;
              const float a = ex2_ftz(m_run - m_new);
#pragma unroll
              for (int e = 0; e < kBN / 4; ++e) pk[e] = scale_pair<DT>(pk[e], a);
              h0 *= a;
              h1 = exp_pairs<DT, ALIBI, kBN / 4, kBN / 2>(s, sl2x2, f2pack(-m_new, -m_new), pk);
            }
            break;
          }
          exact = true;  // a first half failed: redo the row from the tile max
          spec = false;
        }
        need = m_new != m_run && m_new != -INFINITY;
        tsum = h0 + h1;
      } else {
        // level 1: the tile max over the row decides m; level 2: P = 2^(s*sl2 - m)
        const float mt = scaled_max_from<0, ALIBI>(s, sl2);
        need = mt > m_run + kRescaleThreshold;
        m_new = need ? mt : m_run;
        // a row can see no key of this tile (sliding window): keep it at zero weight
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        tsum = exp_pairs<DT, ALIBI, 0, kBN / 2>(s, sl2x2, f2pack(-m_use, -m_use), pk);
      }
      // all exponentials run before any wait below
      const float alpha = need ? ex2_ftz(m_run - m_new) : 1.f;
      if constexpr (C::kSepP) {  // PV_t(j-1) must be done before P_t and O_t are touched
        if (jt > 0) {
          if (!(ok = warp_wait(&bars->pv_done[t], (jt - 1) & 1))) break;
          tc_fence_after();
        }
      }
      if constexpr (C::kSepP) {
        tc_st64(tP, pk);  // one store; measured 1% faster at D = 64
      } else {  // P over S's columns: eight stores measured 0.7% faster at D = 128
#pragma unroll
        for (int cc = 0; cc < kBN / 16; ++cc) tc_st8(tP + 8 * cc, pk + 8 * cc);
      }
      l_run = fmaf(l_run, alpha, tsum);
      // level 3 correction: rescale O in TMEM when some row's max moved
      if (jt > 0 && __any_sync(0xffffffffu, need)) {
        const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
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
    // A sliding window can leave query tile 1 of the last unit without any key
    // tile, when all its rows lie past Nq (every row below Nq sees its own key):
    // then no PV is issued for it and it has nothing to write.
    const bool has_keys = jhi > jlo;
    if (ok && has_keys) ok = warp_wait(&bars->o_final[t], 0);
    if (ok && has_keys) {
      // epilogue: O / l in the output dtype, LSE in natural log
      tc_fence_after();
      const float inv = 1.0f / l_run;
      const bool row_ok = row < Nq;
      if (piece) {  // partial row g of the split tail: O_s and lse_s in fp32
        const long long g = static_cast<long long>(unit - n_full) * (2 * kBM) + (row - r0);
        // the tail holds (gridDim.x - n_full) / n_split units of 2 * kBM partial rows
        const bool in_ws = RF_INB(g < static_cast<long long>(gridDim.x - n_full) / n_split * (2 * kBM) &&
                                      split < n_split, status);
        float4* prow = reinterpret_cast<float4*>(o_part + (g * n_split + split) * D);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          uint32_t ov[32];
          tc_ld32(tO + 32 * i, ov);
          tc_wait_ld();
          if (row_ok && in_ws) {
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              prow[i * 8 + v4] =
                  make_float4(__uint_as_float(ov[4 * v4]) * inv, __uint_as_float(ov[4 * v4 + 1]) * inv,
                              __uint_as_float(ov[4 * v4 + 2]) * inv, __uint_as_float(ov[4 * v4 + 3]) * inv);
          }
        }
        if (row_ok && in_ws) lse_part[g * n_split + split] = (m_run + log2f(l_run)) * kLn2;
      } else {
        // The warp's 32 rows of O are contiguous in memory: they are staged in
        // Q_t's shared-memory tile (free now: every S_t has completed), in the
        // 128-byte swizzle Q arrived in, and written by one TMA store per
        // 64-column box (rows past Nq are clipped); a per-thread store of each
        // row touched 32 lines per instruction.
        const bool in_o = RF_INB(bh < BH && (!row_ok || (row >= 0 && row < Nq)), status);
        uint8_t* ob = sQ + t * C::kQBytes + qw * 32 * 128;  // row `lane` of the warp at ob + lane * 128
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          uint32_t ov[32];
          tc_ld32(tO + 32 * i, ov);
          tc_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = Pack<DT>::pack2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {  // 16-byte chunk gc of the row: box gc / 8, chunk gc mod 8
            const int gc = 4 * i + v4;
            *reinterpret_cast<uint4*>(ob + (gc >> 3) * (kBM * 128) + lane * 128 + ((((gc & 7) ^ lane) & 7) << 4)) =
                make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        fence_proxy_async_smem();  // the staged rows are visible to the TMA store
        __syncwarp();
        const int wrow = row - lane;  // the warp's first row
        if (lane == 0 && wrow < Nq && in_o) {
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx) tma_store_3d(&to, ob + bx * (kBM * 128), bx * 64, wrow, bh);
          tma_store_commit();
          tma_store_wait_read();  // Q_t's tile has been read before the CTA exits; the writes finish on their own
        }
        if (row_ok && in_o && lse) lse[static_cast<long long>(bh) * Nq + row] = (m_run + log2f(l_run)) * kLn2;
      }
    } else if (!ok) {
      if (lane == 0) atomicOr(status, kStatusTimeout);
      bars->abort = 1;
      if (piece && row < Nq) {  // a split-tail piece marks its partial row invalid for the merge
        const long long g = static_cast<long long>(unit - n_full) * (2 * kBM) + (row - r0);
        if (RF_INB(g < static_cast<long long>(gridDim.x - n_full) / n_split * (2 * kBM), status))
          lse_part[g * n_split + split] = NAN;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
}

// Split-tail plan: the last `tail` = units mod sms units become n_split pieces
// each (n_split = min(sms / tail, key tiles) >= 2), else nothing is split.
struct TailPlan {
  long long n_full;
  int tail, n_split;
};

TailPlan tail_plan(long long units, int n_kv, int sms) {
  const int tail = sms > 0 ? static_cast<int>(units % sms) : 0;
  const int n_split = tail > 0 ? min(sms / tail, n_kv) : 1;
  if (tail == 0 || n_split < 2) return TailPlan{units, 0, 1};
  return TailPlan{units - tail, tail, n_split};
}

// Workspace layout of a split tail: o_part [tail * 256, n_split, D] fp32, then
// lse_part [tail * 256, n_split] fp32 at the next 256-byte boundary.
size_t tail_o_bytes(const TailPlan& p, int D) {
  return (static_cast<size_t>(p.tail) * 2 * kBM * p.n_split * D * sizeof(float) + 255) & ~size_t(255);
}
size_t tail_bytes(const TailPlan& p, int D) {
  if (p.tail == 0) return 0;
  return tail_o_bytes(p, D) + static_cast<size_t>(p.tail) * 2 * kBM * p.n_split * sizeof(float);
}

TailPlan plan_for(int B, int Hq, int Nq, int Nk, int sms) {
  const long long units = static_cast<long long>((Nq + 2 * kBM - 1) / (2 * kBM)) * B * Hq;
  return tail_plan(units, (Nk + kBN - 1) / kBN, sms);
}

// The rotary-embedding part of a call: mode 0 none, 1 Q, 2 Q and K.
struct AttnRope {
  int mode = 0;
  int pos = 0;
  double base = 10000.0;
};

template <Dt DT, int D, int MASK, bool ALIBI, int ROPE>
cudaError_t launch_cfg(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, float scale, int window, const float* alibi, unsigned* status,
                       const TailPlan& plan, void* ws, const AttnRope& rp, cudaStream_t s) {
  alignas(64) CUtensorMap tq, tk, tv, to;
  cudaError_t err = cudaSuccess;
  if (!encode_tma_3d_16bit(&tq, q, D, Nq, uint64_t(B) * Hq, kBM, &err)) return err;
  if (!encode_tma_3d_16bit(&to, o, D, Nq, uint64_t(B) * Hq, 32, &err)) return err;  // one warp's rows
  if (!encode_tma_3d_16bit(&tk, k, D, Nk, uint64_t(B) * Hkv, kBN, &err)) return err;
  if (!encode_tma_3d_16bit(&tv, v, D, Nk, uint64_t(B) * Hkv, kBN, &err)) return err;
  const int nqt = (Nq + 2 * kBM - 1) / (2 * kBM);
  const long long grid = static_cast<long long>(nqt) * B * Hq;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int smem = Cfg<D>::kTiles + (ROPE == 2 ? Cfg<D>::kRopeBytes : 0) + 1024 + static_cast<int>(sizeof(TcBars)) + 64;
  auto kern = attn_tc_kernel<DT, D, MASK, ALIBI, ROPE>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  RopeParams rope{};
  if (ROPE) rope = make_rope_params(rp.base, D);
  // Causal units run longest first with every head of one query-tile index
  // adjacent, so the K and V tiles of all heads are reused through L2.  When
  // they take much of L2 (with Q and O streaming past them) they get evicted
  // and re-read: then the batches run one after another instead.  Measured: K
  // and V of 67 MB (B=2 Hq=32 Hkv=8 N=8192 D=128) were re-read, DRAM reads
  // 365 -> 204 MB and 0.8% faster batch-major; 50 MB (B=4 H=12 N=4096 D=64)
  // stayed in L2, and batch-major was 2.8% slower there.  The threshold, 45%
  // of L2, lies between the two.
  const long long kv_bytes = 2LL * B * Hkv * Nk * D * 2;
  const int batch_major = MASK >= 1 && B > 1 && kv_bytes * 20 > device_l2_bytes() * 9 ? 1 : 0;
  const bool split = MASK == 0 && plan.tail > 0 && ws != nullptr;
  float* o_part = split ? static_cast<float*>(ws) : nullptr;
  float* lse_part = split ? reinterpret_cast<float*>(static_cast<char*>(ws) + tail_o_bytes(plan, D)) : nullptr;
  const long long n_full = split ? plan.n_full : grid;
  const long long ctas = split ? plan.n_full + static_cast<long long>(plan.tail) * plan.n_split : grid;
  kern<<<static_cast<unsigned>(ctas), kThreads, smem, s>>>(tq, tk, tv, to, lse, Hq, Hkv, Nq,
                                                           Nk, B * Hq, nqt, scale * kLog2e, window, alibi, status,
                                                           static_cast<int>(n_full), split ? plan.n_split : 1,
                                                           o_part, lse_part, rope, rp.pos, batch_major,
                                                           D == 128 ? device_sm_count() : 0);
  err = cudaGetLastError();
  if (err != cudaSuccess || !split) return err;
  const int rows = plan.tail * 2 * kBM;
  const AttnTailRows map{static_cast<int>(plan.n_full), B * Hq, nqt, Nq};
  // Launched with programmatic stream serialisation: its launch overlaps the
  // attention grid's last wave, and it waits on the device for that grid.
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps));
  lc.blockDim = dim3(kMergeWarps * 32);
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = la;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, lse_merge_kernel<DT, AttnTailRows>, static_cast<const float*>(o_part),
                            static_cast<const float*>(lse_part), o, lse, rows, plan.n_split, D, map,
                            static_cast<long long>(B) * Hq * Nq, status);
}

// One head dimension and rotary mode: the mask and ALiBi pick the instance
// (the rotary modes are built without ALiBi).
template <Dt DT, int D, int ROPE>
cudaError_t launch_d(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, float scale, int causal, int window, const float* alibi, unsigned* status,
                     const TailPlan& plan, void* ws, const AttnRope& rp, cudaStream_t s) {
  const TailPlan none{0, 0, 1};
  if (!causal)
    return launch_cfg<DT, D, 0, false, ROPE>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, 0, nullptr, status, plan,
                                             ws, rp, s);
  if constexpr (ROPE == 0) {
    if (alibi && window > 0)
      return launch_cfg<DT, D, 2, true, 0>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, window, alibi, status, none,
                                           nullptr, rp, s);
    if (alibi)
      return launch_cfg<DT, D, 1, true, 0>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, 0, alibi, status, none,
                                           nullptr, rp, s);
  } else {
    if (alibi) return cudaErrorNotSupported;
  }
  if (window > 0)
    return launch_cfg<DT, D, 2, false, ROPE>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, window, nullptr, status,
                                             none, nullptr, rp, s);
  return launch_cfg<DT, D, 1, false, ROPE>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, 0, nullptr, status, none,
                                           nullptr, rp, s);
}

// Every dtype and head dimension of one rotary mode.
template <int ROPE>
cudaError_t launch_rope_mode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Nq, int Nk, int D, float scale, int causal, int window, const float* alibi,
                             Dt dt, unsigned* status, void* ws, int sms, const AttnRope& rp, cudaStream_t s) {
  const TailPlan plan = plan_for(B, Hq, Nq, Nk, sms);
#define RF_ATTN_ARGS q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, alibi, status, plan, ws, rp, s
  if (dt == Dt::BF16)
    return D == 128 ? launch_d<Dt::BF16, 128, ROPE>(RF_ATTN_ARGS) : launch_d<Dt::BF16, 64, ROPE>(RF_ATTN_ARGS);
  if (dt == Dt::F16)
    return D == 128 ? launch_d<Dt::F16, 128, ROPE>(RF_ATTN_ARGS) : launch_d<Dt::F16, 64, ROPE>(RF_ATTN_ARGS);
#undef RF_ATTN_ARGS
  return cudaErrorNotSupported;
}

}  // namespace
}  // namespace rf
