/*
 * rf.h -- C ABI of librf.so: fused cascaded reductions on one GB300 (sm_103a).
 *
 * A cascaded reduction is a chain of reductions over one input stream where
 * each level depends on the results of the levels before it (RedFuser: An
 * Automatic Operator Fusion Framework for Cascaded Reductions on AI
 * Accelerators, Abstract; Figures 1-2).  Every call below evaluates such a
 * chain in one pass over its input, in the incremental form of RedFuser's
 * Figure 4: as each block of input arrives, every level's running result is
 * updated and the earlier levels' results are corrected with the combine
 * operator that distributes over the reduce operator (RedFuser, Table 1:
 * max with +, + with *).  The input is read from HBM once and the on-chip
 * state has a constant size.
 *
 * Conventions shared by all calls
 * -------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller, contiguous
 *   row-major in the layout stated at each call.  The library allocates no
 *   device memory; the one call that needs scratch takes it from the caller
 *   (rf_attn_decode_splitkv's workspace), and its _noalloc variant uses a
 *   fixed scratch array built into the library instead.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls are asynchronous: they enqueue kernels on `stream` and
 *   return; results are ready once the stream has been synchronised, and work
 *   the caller enqueues after a call in the ordinary way starts after it.
 *   The attention and split-KV decode kernels allow programmatic dependent
 *   launch (they signal griddepcontrol.launch_dependents once set up, which
 *   lets their own merge kernel start early): a kernel the caller launches
 *   next with programmatic stream serialisation may start before the call's
 *   outputs are written, and must wait (cudaGridDependencySynchronize) before
 *   it reads them, as programmatic dependent launch requires in general.
 * - `dtype` names the element type of the 16/32-bit tensors; accumulation is
 *   always fp32.  Softmax scores use natural exponentials; LSE outputs are
 *   natural logarithms of sum_j exp(scale * q.k_j).
 * - Argument checks run on the host before anything is enqueued.  A failing
 *   check returns an error status, leaves every output untouched and records a
 *   message that rf_last_error() returns (per host thread).  No call aborts the
 *   process, and no kernel traps: a device-side wait that runs out of its
 *   iteration budget records RF_ERR_TIMEOUT in a device status word that
 *   rf_device_status() reports.
 */
#ifndef RF_H_
#define RF_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RF_VERSION 10100 /* 1.1.0 */

typedef enum {
  RF_OK = 0,
  RF_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, short workspace */
  RF_ERR_UNSUPPORTED = 2,  /* well-formed but not implemented (e.g. head dim) */
  RF_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  RF_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out (rf_device_status) */
  RF_ERR_CHECK = 5         /* an index check of a checked build failed (rf_device_status) */
} rf_status_t;

typedef enum { RF_F32 = 0, RF_F16 = 1, RF_BF16 = 2 } rf_dtype_t;

/*
 * rf_attn_fwd -- attention forward, the cascade max -> sum exp -> sum exp*v.
 *
 * Defines O = softmax(scale * Q K^T + mask) V per (batch, query head), the
 * "safe softmax followed by GEMM" of RedFuser's Abstract and the attention
 * fusion pattern of the "Operator Fusion" guide (section 2, Pattern 4), with
 * level 1 the running row max, level 2 the running sum of exp(s - max) and
 * level 3 the running exp-weighted sum of V, each rescaled by
 * exp(max_old - max_new) when a key block raises the max.
 *
 *   q    [B, Hq,  Nq, D]  dtype          (read)
 *   k, v [B, Hkv, Nk, D]  dtype          (read)
 *   o    [B, Hq,  Nq, D]  dtype          (written)
 *   lse  [B, Hq,  Nq]     fp32, nullable (written: max + ln(sum exp), natural log)
 *   Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention
 *   with consecutive groups).  causal != 0 applies the top-left lower-triangular
 *   mask (key j visible to query i iff j <= i) and requires Nq == Nk.
 *
 * Supported: dtype RF_F16 / RF_BF16 with D in {64, 128} (tcgen05 tensor-core
 * kernel); dtype RF_F32 with D a multiple of 4, 4 <= D <= 128 (exact fp32 SIMT
 * kernel).  Pointers must be 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG for null q/k/v/o, B/Hq/Hkv/Nq/Nk/D <= 0,
 * Hq % Hkv != 0, misalignment or a non-finite/non-positive scale;
 * RF_ERR_UNSUPPORTED for other D, or causal with Nq != Nk; RF_ERR_CUDA if the
 * launch fails.
 */
rf_status_t rf_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                        int causal, rf_dtype_t dtype, void* stream);

/*
 * rf_attn_fwd_ex -- rf_attn_fwd with score variants (AttnFuse, Table 6: a
 * sliding window W=256 and causal + ALiBi beside dense and causal).
 *
 * Options (opts nullable = non-causal, no variant):
 *   causal        top-left causal mask; requires Nq == Nk.
 *   window        > 0: a key j is also hidden from query i unless
 *                 j > i - window (the window counts the query's own key).
 *                 Key tiles wholly outside every row's window are skipped.
 *                 With 16-bit inputs at D = 64, windows of up to 1024 keys run
 *                 on a persistent kernel (one CTA per SM walking units of 256
 *                 query rows); the results are the same either way.
 *   alibi_slopes  nullable device pointer to Hq fp32 slopes: slope[h]*(j - i)
 *                 is added to each scaled score (the linear-bias form of ALiBi).
 *   workspace     nullable device memory of workspace_bytes bytes (16-byte
 *                 aligned, owned by the caller, contents need not be set).
 *                 Without a mask, the 16-bit kernel runs one CTA of 256 query
 *                 rows per SM; when the last wave of such units is short, a
 *                 workspace lets those units be split along the keys over the
 *                 idle SMs and merged by a log-sum-exp combine (RedFuser,
 *                 Figure 13: the FlashDecoding split and merge) in a second
 *                 kernel on the same stream.  It needs
 *                 rf_attn_fwd_workspace_bytes(...) bytes; a null workspace
 *                 runs every unit whole (same results up to rounding order).
 *                 Calls that overlap on the GPU must not share a workspace.
 *   rope          rotary position embedding fused into the load (AttnFuse,
 *                 Figure 1 and Table 4): the pair (x_i, x_{i+D/2}) of a row at
 *                 position p turns by p * rope_base^(-2i/D), with
 *                 p = rope_pos_offset + row index.  1 turns the Q rows once per
 *                 CTA after their load (for K already rotated, e.g. a cached
 *                 K); 2 also turns the K rows of every key tile, which every
 *                 CTA that streams the tile repeats.  q, k and v are not
 *                 modified.  The result equals attention over the rows that
 *                 rf_rope_qk writes (Q bit for bit; K up to the rounding of
 *                 its angles' cosines and sines).  16-bit paths only, without
 *                 ALiBi (RF_ERR_UNSUPPORTED otherwise); positions must stay
 *                 below 2^24; rope outside {0, 1, 2}, a negative offset or a
 *                 base that is negative, 1 or not finite is RF_ERR_INVALID_ARG.
 *                 Callers should zero the whole struct before setting fields:
 *                 versions before 1.1.0 do not have these three.
 * The window and ALiBi need the causal mask (RF_ERR_UNSUPPORTED otherwise).
 * The LSE output includes the ALiBi bias.  Everything else (layouts,
 * supported dtypes and head dims, errors) is as rf_attn_fwd; a negative window
 * is RF_ERR_INVALID_ARG, and so is a workspace smaller than it needs to be.
 */
typedef struct rf_attn_opts_t {
  int causal;
  int window;
  const float* alibi_slopes;
  void* workspace;        /* nullable device memory, see rf_attn_fwd_workspace_bytes */
  size_t workspace_bytes;
  /* since version 1.1.0: rotary embedding applied inside the kernel */
  int rope;               /* 0 none, 1 rotate the Q rows, 2 rotate the Q and K rows */
  float rope_base;        /* angle base; 0 means 10000 */
  int rope_pos_offset;    /* position of query row 0 and of key 0 (>= 0) */
} rf_attn_opts_t;
rf_status_t rf_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                           const rf_attn_opts_t* opts, rf_dtype_t dtype, void* stream);

/*
 * rf_attn_fwd_workspace_bytes -- bytes of workspace that rf_attn_fwd_ex can
 * use for the split of the last short wave on the current device (its
 * multiprocessor count decides the split).  0 when nothing would be split:
 * causal, fp32, a single key tile, or a last wave that is full or more than
 * half full.  (size_t)-1 for invalid sizes, an unsupported D, or a device that
 * cannot be queried.  At most 256 rows x (D + 1) x 4 bytes per multiprocessor
 * (about 20 MiB on 152 SMs at D = 128).
 */
size_t rf_attn_fwd_workspace_bytes(int B, int Hq, int Nq, int Nk, int D, int causal, rf_dtype_t dtype);

/*
 * rf_attn_decode_splitkv_workspace_bytes -- scratch size for rf_attn_decode_splitkv:
 * fp32 partial outputs [B*Hq, num_splits, D] followed (at a 256-byte aligned
 * offset) by fp32 partial LSEs [B*Hq, num_splits].  Returns 0 for non-positive
 * arguments.
 */
size_t rf_attn_decode_splitkv_workspace_bytes(int B, int Hq, int D, int num_splits);

/*
 * rf_attn_decode_splitkv -- one decoding step (one query per head) over a KV
 * cache, split along the keys and merged by log-sum-exp (split-KV or "flash"
 * decoding: RedFuser, Figure 13 "FlashDecoding IR"; AttnFuse, Table 8).
 *
 * Split s covers the contiguous keys [floor(s*L/S), floor((s+1)*L/S)).  For
 * each (batch, kv head, split) one CTA runs the fused cascade for all
 * G = Hq/Hkv query heads of the group and writes the split's normalised O_s
 * and lse_s into the workspace; a second kernel on the same stream merges the
 * splits (the same combine as rf_lse_merge).  An empty split (L < S) has
 * lse_s = -inf and weight 0.
 *
 *   q        [B, Hq, D]        dtype  (read; one query per head)
 *   k_cache  [B, Hkv, L, D]    dtype  (read)
 *   v_cache  [B, Hkv, L, D]    dtype  (read)
 *   o        [B, Hq, D]        dtype  (written)
 *   lse      [B, Hq]           fp32, nullable (written)
 *   workspace: device scratch of at least
 *     rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits) bytes,
 *     256-byte aligned, caller-owned; its contents after the call are the
 *     per-split partials (layout as documented at the size query).
 *
 * Supported: dtype RF_F16 / RF_BF16, D in {64, 128}, 1 <= Hq/Hkv <= 8,
 * 1 <= num_splits <= 256.  Pointers 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG for null pointers, non-positive sizes,
 * Hq % Hkv != 0, misalignment, or a short workspace; RF_ERR_UNSUPPORTED for
 * other dtype / D / group size; RF_ERR_CUDA if a launch fails.  A split whose
 * bounded wait runs out (reported later by rf_device_status as
 * RF_ERR_TIMEOUT) writes NaN partials, so the rows it feeds come out NaN.
 */
rf_status_t rf_attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                                   void* o, float* lse, void* workspace, size_t workspace_bytes,
                                   int B, int Hq, int Hkv, int L, int D, int num_splits,
                                   float scale, rf_dtype_t dtype, void* stream);

/*
 * rf_attn_decode_splitkv_noalloc -- rf_attn_decode_splitkv without a
 * workspace argument, for callers that cannot allocate device memory: for
 * example a plugin whose host framework owns all device memory and hands it
 * only the input and output buffers, or a serving loop that reserves all its
 * memory at start-up and forbids later allocation because cudaMalloc can
 * synchronise the device and can fail under memory pressure mid-run.  The
 * pages describe no such call; it exists for this deployment constraint only.
 *
 * Same arguments, layouts, results and errors as rf_attn_decode_splitkv,
 * minus `workspace` / `workspace_bytes`.  The per-split partials live in a
 * scratch array of RF_DECODE_NOALLOC_SCRATCH_BYTES built into the library
 * (every GPU that loads the library holds it until the process exits).
 * - Sizes whose partials need more than that (see
 *   rf_attn_decode_splitkv_workspace_bytes) return RF_ERR_INVALID_ARG with a
 *   message naming both sizes; no kernel is launched.
 * - The call allocates nothing (no cudaMalloc, no cudaFree).  Its first call
 *   on each device looks up the scratch address with cudaGetSymbolAddress
 *   (with that device current); make that first call before any stream
 *   capture.
 * - All calls share the one scratch array: calls that can overlap on the GPU
 *   (other streams, other host threads) race on it and must be serialised by
 *   the caller.  After a call the array holds that call's partials (NaN for
 *   a split whose bounded wait ran out, which also makes its rows' outputs
 *   NaN); nothing in it needs to start at zero.
 */
#define RF_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */
rf_status_t rf_attn_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                           void* o, float* lse, int B, int Hq, int Hkv, int L, int D,
                                           int num_splits, float scale, rf_dtype_t dtype, void* stream);

/*
 * rf_lse_merge -- combine partial attention results computed over disjoint
 * key sets: LSE = ln sum_s exp(lse_s), O = sum_s exp(lse_s - LSE) * O_s.
 * This is the incremental combine across splits (RedFuser, Figure 4 and
 * Figure 13): level 2 (sum, combine *) rebuilt from the parts' LSEs, level 3
 * rescaled by the same weights.
 *
 *   o_part   [rows, num_splits, D] fp32 (read; normalised partial outputs)
 *   lse_part [rows, num_splits]    fp32 (read; -inf marks an empty part)
 *   o        [rows, D]             out_dtype (written)
 *   lse      [rows]                fp32, nullable (written)
 *   A row whose parts are all empty gets O = 0 and LSE = -inf.  A part whose
 *   lse_s is NaN (a split that gave up after a bounded wait writes that) makes
 *   the row's O and LSE NaN.  Each weight is formed as exp(lse_s - max) / sum
 *   over the row's parts, so the rounding of LSE does not enter the weights.
 *
 * Supported: out_dtype RF_F32 / RF_F16 / RF_BF16, D a multiple of 4 up to 512,
 * 1 <= num_splits <= 256.  o_part and o 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG for null inputs/outputs, non-positive sizes or
 * misalignment; RF_ERR_UNSUPPORTED for D or num_splits out of range;
 * RF_ERR_CUDA if the launch fails.
 */
rf_status_t rf_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                         int rows, int num_splits, int D, rf_dtype_t out_dtype, void* stream);

/*
 * rf_layernorm_fused -- residual add + LayerNorm in one pass over each row:
 * h = x + residual; mean and biased variance of h from running sums of
 * (h - K) and (h - K)^2 about K, the mean of the row's first 16-byte vector,
 * merged across threads by addition (a row whose K lies more than one standard
 * deviation from its mean recomputes the variance about the mean from the
 * values it holds); y = ((h - K) - (mean - K)) / sqrt(var + eps) * gamma + beta
 * ("Operator Fusion" guide, section 1 and section 2 Pattern 2; section 4
 * places eps inside the root).
 * The row is kept on chip between the statistics and the normalisation, so
 * x and residual are read once and y written once.
 *
 *   x, residual   [rows, cols] dtype (read; residual nullable = no residual add)
 *   gamma, beta   [cols]       dtype (read; nullable = 1 and 0)
 *   out           [rows, cols] dtype (written)
 *   residual_out  [rows, cols] dtype, nullable (written: h rounded to dtype)
 *
 * Supported: dtype RF_F32 / RF_F16 / RF_BF16; cols a multiple of 16 bytes'
 * worth of elements (8 for 16-bit, 4 for fp32) and at most 32768 (16-bit) or
 * 16384 (fp32); all pointers 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG for null x/out, non-positive sizes, eps < 0 or
 * misalignment; RF_ERR_UNSUPPORTED for cols out of range; RF_ERR_CUDA if the
 * launch fails.
 */
rf_status_t rf_layernorm_fused(const void* x, const void* residual, const void* gamma,
                               const void* beta, void* out, void* residual_out,
                               int rows, int cols, float eps, rf_dtype_t dtype, void* stream);

/*
 * rf_rmsnorm_fused -- residual add + RMSNorm in one pass over each row:
 * h = x + residual; the one reduction level is the running sum of squares of
 * h (combine op +); y = h * gamma / sqrt(sum(h^2)/cols + eps).  The
 * "Operator Fusion" guide (section 3) lists RMSNorm with LayerNorm as a
 * fusible reduction + normalise pattern; eps sits inside the root as in its
 * LayerNorm kernels, and there is no bias.  The row stays on chip between
 * the reduction and the normalisation (x and residual read once, y written
 * once).
 *
 *   x, residual   [rows, cols] dtype (read; residual nullable)
 *   gamma         [cols]       dtype (read; nullable = 1)
 *   out           [rows, cols] dtype (written)
 *   residual_out  [rows, cols] dtype, nullable (written: h rounded to dtype)
 *
 * Supported sizes, alignment and errors: as rf_layernorm_fused.
 */
rf_status_t rf_rmsnorm_fused(const void* x, const void* residual, const void* gamma, void* out,
                             void* residual_out, int rows, int cols, float eps, rf_dtype_t dtype,
                             void* stream);

/*
 * rf_softmax_xent -- fused softmax + cross-entropy per row of logits, the
 * cascade max -> sum exp -> loss ("Operator Fusion" guide, section 3: softmax
 * + cross-entropy is fusible).  Level 1 is the running row max, level 2 the
 * running sum of exp(z - max), rescaled whenever the max rises (RedFuser's
 * incremental form); loss = max + ln(sum) - z[target].  Logits are read once.
 *
 *   logits  [rows, vocab] dtype      (read)
 *   targets [rows]        int64      (read; class index, or ignore_index)
 *   loss    [rows]        fp32       (written; 0 for an ignored row, NaN for a
 *                                     target outside [0, vocab))
 *   lse     [rows]        fp32, nullable (written: natural-log sum exp)
 *   grad    [rows, vocab] dtype, nullable (written: softmax(z) - onehot(target),
 *                                     unscaled; all zero for an ignored row)
 *
 * Supported: dtype RF_F32 / RF_F16 / RF_BF16; vocab a multiple of 16 bytes'
 * worth of elements (8 for 16-bit, 4 for fp32); logits and grad 16-byte
 * aligned.  Many rows run one CTA per row; fewer rows than multiprocessors
 * run each row on a thread-block cluster of up to 8 CTAs that merge their
 * partial (max, sum exp) through distributed shared memory.  Any rows >= 1.
 * Errors: RF_ERR_INVALID_ARG for null logits/targets/loss, non-positive sizes,
 * misalignment or a vocab that is not a whole number of vectors; RF_ERR_CUDA
 * if the launch fails.
 */
rf_status_t rf_softmax_xent(const void* logits, const long long* targets, float* loss, float* lse, void* grad,
                            int rows, int vocab, long long ignore_index, rf_dtype_t dtype, void* stream);

/*
 * rf_rope_qk -- rotary position embedding of Q and K, the pre-matmul
 * transformation of AttnFuse (Abstract; Figure 1), as one HBM pass ahead of
 * the attention call.  For i < D/2 the pair (x_i, x_{i+D/2}) of the row at
 * position p = pos_offset + n turns by theta = p * base^(-2i/D):
 *   y_i = x_i cos theta - x_{i+D/2} sin theta,
 *   y_{i+D/2} = x_i sin theta + x_{i+D/2} cos theta  (rotate-half pairing).
 *
 *   q      [B, Hq, N, D]  dtype (read)        q_out  [B, Hq, N, D]  (written)
 *   k      [B, Hkv, N, D] dtype (read)        k_out  [B, Hkv, N, D] (written)
 * k and k_out are both null (rotate Q only) or both non-null.  An output may
 * be its own input (in place).  Angles are formed to about 1e-7 rad for any
 * position below 2^24 and reduced to [-pi, pi]; their cosines and sines come
 * from the hardware functions, accurate to a few 1e-7 there.  The rotation
 * inside rf_attn_fwd_ex (rope = 1) uses the same function, bit for bit.
 *
 * Supported: dtype RF_F16 / RF_BF16; D in {64, 128, 256}; base > 0, finite,
 * not 1; pos_offset >= 0 and pos_offset + N <= 2^24; pointers 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG for null q/q_out, a k without k_out (or the
 * reverse), non-positive sizes, a bad base or offset, misalignment;
 * RF_ERR_UNSUPPORTED for other D or dtypes and positions past 2^24;
 * RF_ERR_CUDA if the launch fails.
 */
rf_status_t rf_rope_qk(const void* q, const void* k, void* q_out, void* k_out, int B, int Hq, int Hkv, int N, int D,
                       float base, int pos_offset, rf_dtype_t dtype, void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* rf_last_error(void);

/* RF_VERSION of the loaded library. */
int rf_version(void);

/*
 * rf_checks_enabled -- 1 when the library was built with -DRF_CHECKS, else 0.
 * In such a build every kernel checks the indices it computes (tensor
 * coordinates, output rows and offsets, split-tail and workspace slots, shared
 * memory tiles) before it uses them; a check that fails skips the access,
 * never traps, and records RF_ERR_CHECK for rf_device_status.  The checks run
 * inside the kernels, at full size, with no external tool.
 */
int rf_checks_enabled(void);

/*
 * rf_selftest_check -- launches one thread that evaluates an index check
 * which always fails, without touching memory: in a checked build the device
 * status word then reports RF_ERR_CHECK (rf_device_status); in other builds
 * nothing is recorded.  RF_ERR_CUDA if the launch fails.
 */
rf_status_t rf_selftest_check(void* stream);

/*
 * rf_device_status -- synchronise `stream`, then report whether any kernel of
 * this library on the current device recorded a failed index check
 * (RF_ERR_CHECK, checked builds only) or else a bounded wait that ran out
 * (RF_ERR_TIMEOUT) since the status was last cleared; clear != 0 resets it.
 * Returns RF_ERR_CUDA if the synchronisation itself fails.
 */
rf_status_t rf_device_status(void* stream, int clear);

/*
 * rf_selftest_wait_timeout -- exercise the failure path of the bounded
 * device-side waits: launch one warp that waits on a barrier nothing signals,
 * gives up after timeout_us microseconds (1 .. 1,000,000), and records
 * RF_ERR_TIMEOUT in the device status word, as a production kernel does when
 * one of its waits runs out.  No copy or tensor-memory allocation is in flight
 * when it gives up, so the context stays usable.  A following
 * rf_device_status() returns RF_ERR_TIMEOUT (and clears it when asked).
 * Errors: RF_ERR_INVALID_ARG for a timeout out of range; RF_ERR_CUDA if the
 * launch fails.
 */
rf_status_t rf_selftest_wait_timeout(unsigned timeout_us, void* stream);

/*
 * Ablation variants of the fused cascades (RedFuser, Figure 6: (a) fusion at
 * different levels, (b) incremental vs non-incremental computation; Figure 7:
 * what each level of fusion saves in re-reads).  These entry points exist to
 * measure what the fused incremental kernels gain; they compute the same
 * results, differing only in rounding order.
 *
 * rf_layernorm_ablation -- residual + LayerNorm as rf_layernorm_fused (x,
 * residual, gamma, beta all required; no residual_out) with `variant`:
 *   0  fused, incremental: rf_layernorm_fused itself (one read of x and r).
 *   1  fused, non-incremental: one CTA per row stages h = x + r in shared
 *      memory (cols * 4 bytes of on-chip memory), then a mean pass, a
 *      variance pass and a normalise pass over it.  cols <= 56,832.
 *   2  reductions fused, normalise separate: one kernel reads x and r for
 *      (mean, rstd) per row; a second kernel reads x and r again to normalise.
 *   3  unfused: h = x + r written to HBM, then a mean kernel, a variance kernel
 *      and a normalise kernel, each reading h from HBM.
 * rf_softmax_xent_ablation -- loss (and lse) as rf_softmax_xent without the
 * gradient, with `variant`:
 *   0  fused, incremental: rf_softmax_xent itself (one read of the logits).
 *   1  fused, two-pass: one CTA per row reads the row for the max, then again
 *      for sum exp(z - max) (level 2 waits for all of level 1; the row would
 *      not fit on chip at vocabulary sizes, so the second pass re-reads it).
 *   2  unfused: a max kernel, a sum-of-exponentials kernel and a loss kernel.
 *
 * `workspace` is device memory of at least rf_ablation_workspace_bytes(op,
 * variant, rows, cols, dtype) bytes (op 0 = LayerNorm, 1 = cross-entropy;
 * cols = vocab for op 1), 256-byte aligned, owned by the caller; nullable
 * when that size is 0.  rf_ablation_workspace_bytes returns 0 for a variant
 * that needs none and (size_t)-1 for invalid arguments.
 * Errors: as the fused entry points, plus RF_ERR_INVALID_ARG for an unknown
 * variant or a missing/short workspace and RF_ERR_UNSUPPORTED for a row too
 * long for variant 1's shared memory.
 */
size_t rf_ablation_workspace_bytes(int op, int variant, int rows, int cols, rf_dtype_t dtype);
rf_status_t rf_layernorm_ablation(const void* x, const void* residual, const void* gamma, const void* beta,
                                  void* out, int rows, int cols, float eps, int variant, void* workspace,
                                  size_t workspace_bytes, rf_dtype_t dtype, void* stream);
rf_status_t rf_softmax_xent_ablation(const void* logits, const long long* targets, float* loss, float* lse,
                                     int rows, int vocab, long long ignore_index, int variant, void* workspace,
                                     size_t workspace_bytes, rf_dtype_t dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RF_H_ */
