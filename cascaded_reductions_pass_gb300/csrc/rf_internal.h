// Host-side declarations shared by the ABI front end (rf_api.cu) and the
// kernel translation units.  Every launcher enqueues on `stream`, performs no
// allocation and returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rf {

enum class Dt : int { F32 = 0, F16 = 1, BF16 = 2 };

// residual + LayerNorm (ln_fused.cu)
int layernorm_max_cols(Dt dt);
cudaError_t launch_layernorm(const void* x, const void* r, const void* gamma, const void* beta,
                             void* out, void* r_out, int rows, int cols, float eps, Dt dt,
                             unsigned* status, cudaStream_t s);

// residual + RMSNorm (ln_fused.cu; same limits as LayerNorm)
cudaError_t launch_rmsnorm(const void* x, const void* r, const void* gamma, void* out, void* r_out, int rows,
                           int cols, float eps, Dt dt, unsigned* status, cudaStream_t s);

// softmax cross-entropy per row, optional gradient (xent_fused.cu)
cudaError_t launch_xent(const void* logits, const long long* targets, float* loss, float* lse, void* grad, int rows,
                        int vocab, long long ignore_index, Dt dt, unsigned* status, cudaStream_t s);

// log-sum-exp merge of split partials (lse_merge.cu); after_split: launched
// right after the kernel that writes the partials, which lets it be scheduled
// early (programmatic dependent launch; the merge waits for that kernel)
cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                             int rows, int splits, int D, Dt out_dt, unsigned* status, cudaStream_t s,
                             bool after_split = false);

// exact fp32 SIMT attention forward (attn_fwd_f32.cu)
cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                            int window, const float* alibi, unsigned* status, cudaStream_t s);

// split-KV decode partials (decode_split.cu): writes o_part [B*Hq, S, D] and
// lse_part [B*Hq, S] fp32.
cudaError_t launch_decode_split(const void* q, const void* k, const void* v, float* o_part,
                                float* lse_part, int B, int Hq, int Hkv, int L, int D, int splits,
                                float scale, Dt dt, unsigned* status, cudaStream_t s);

// tcgen05 / TMEM / TMA attention forward for 16-bit inputs (attn_fwd_tc.cu).
// Without a mask, and with `ws` non-null, the units of the last partial wave
// on `sms` SMs are split along the keys and merged; ws must then hold
// attn_tc_workspace_bytes(...) bytes (0 when nothing is split).
size_t attn_tc_workspace_bytes(int B, int Hq, int Nq, int Nk, int D, int causal, int sms);
// rope: 0 none, 1 rotary embedding of the Q rows inside the kernel, 2 of the Q
// and K rows (positions rope_pos + row, angles base^(-2i/D) with base rope_base).
cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                           int window, const float* alibi, Dt dt, unsigned* status, void* ws, int sms,
                           int rope, double rope_base, int rope_pos, cudaStream_t s);
// the rotary modes 1 and 2 of launch_attn_tc (attn_fwd_tc_rope.cu); no ALiBi
cudaError_t launch_attn_tc_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                                const float* alibi, Dt dt, unsigned* status, void* ws, int sms, int rope,
                                double rope_base, int rope_pos, cudaStream_t s);

// causal sliding-window attention at D = 64 for 16-bit inputs as a persistent
// kernel, one CTA per SM walking a list of 256-row units (attn_fwd_tc_window.cu);
// with sms <= 0, one CTA per unit.  launch_attn_tc sends windows of up to
// kWindowPersistMax keys there.
constexpr int kWindowPersistMax = 1024;
cudaError_t launch_attn_tc_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Nq, int Nk, float scale, int window, const float* alibi, Dt dt,
                                  unsigned* status, int sms, cudaStream_t s);

// multiprocessor count of the current device (cached per device; 0 on error)
int device_sm_count();
// L2 cache size in bytes of the current device (cached per device; 0 on error)
long long device_l2_bytes();

// bounded-wait failure path self-test (selftest.cu)
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned* status, int* waited_out, cudaStream_t s);
// an index check that always fails, with no memory access (selftest.cu)
cudaError_t launch_check_selftest(unsigned* status, cudaStream_t s);

// fusion-level / incremental-form ablation variants (ablation.cu)
constexpr int kLnSmemMaxCols = 56832;  // variant 1 stages cols floats in shared memory
size_t ablation_ln_workspace_bytes(int rows, int cols, int variant, Dt dt);
size_t ablation_xent_workspace_bytes(int rows, int variant);
cudaError_t launch_ln_ablation(const void* x, const void* r, const void* g, const void* b, void* out, int rows,
                               int cols, float eps, int variant, void* ws, Dt dt, cudaStream_t s);
cudaError_t launch_xent_ablation(const void* logits, const long long* targets, float* loss, float* lse, int rows,
                                 int vocab, long long ignore, int variant, void* ws, Dt dt, cudaStream_t s);

// rotary position embedding of Q and K rows, one HBM pass (rope.cu); 16-bit,
// D in {64, 128, 256}; q_out / k_out may alias q / k
constexpr int kRopeMaxHalf = 128;
cudaError_t launch_rope_qk(const void* q, const void* k, void* q_out, void* k_out, int BHq, int BHkv, int N, int D,
                           double base, int pos_offset, Dt dt, unsigned* status, cudaStream_t s);

// TMA descriptor encoding through the driver entry point (rf_api.cu).
// 3-D tensor [outer][rows][inner] of 16-bit elements, box {64, box_rows, 1},
// 128-byte swizzle; returns false (and sets *err) on failure.
bool encode_tma_3d_16bit(void* tmap_out, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t outer, uint32_t box_rows, cudaError_t* err);

}  // namespace rf
