"""Plain fp64 definitions of the cascaded reductions (test infrastructure only).

Citations name the page and the part of it that each step follows:

* RedFuser: An Automatic Operator Fusion Framework for Cascaded Reductions on
  AI Accelerators (thelatestinai.com/papers/2603.10026) -- Abstract ("safe
  softmax followed by GEMM"), Table 1 (reduce/combine operator pairs),
  Figure 13 ("FlashDecoding IR", body not extracted).
* AttnFuse: A Composable DSL for Compiling Attentions to Fused GPU Kernels
  (thelatestinai.com/papers/2609.13612) -- Table 8 ("Flash Decoding", one query
  per head, GQA geometries).
* Operator Fusion (infra.bea.ai/guide/cuda/core-kernels/operator-fusion) --
  section 2 Patterns 2 and 4, section 4 "Manual (CUDA)".

Readings of points the pages leave open (variance divisor, causal alignment,
GQA head map, split partition, LSE base) are stated at each function.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(a):
    """Upcast exactly to float64 (accepts numpy arrays or CPU torch tensors)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").float().numpy()
    return np.asarray(a, dtype=np.float64)


def attention(q, k, v, scale, causal=False, rows=None, window=0, alibi_slopes=None):
    """Plain attention forward: O = softmax(scale * Q K^T [+ mask]) V, and LSE.

    Follows the unfused listing of "Operator Fusion", section 2, Pattern 4:
    scores = Q K^T * scale; mask; softmax; weighted sum of V.  The softmax is
    the *safe* one named in the RedFuser abstract: the row maximum m is taken
    first (level 1, reduce op max), then l = sum_j exp(s_j - m) (level 2, reduce
    op +), then sum_j exp(s_j - m) v_j (level 3, reduce op +), then O = that / l.

    Shapes: q [B,Hq,Nq,D]; k, v [B,Hkv,Nk,D] (v may have its own last dim).
    Readings: query head h reads key/value head h // (Hq/Hkv) (consecutive
    groups); the causal mask is top-left aligned, key j visible to query i iff
    j <= i; LSE_i = m_i + ln l_i in natural log with the scale included.  A row
    with no visible key (Nk == 0) yields O = 0 and LSE = -inf.

    ``rows`` optionally restricts the computation to a list of query indices
    (used for sampled checks at full size); outputs then have len(rows) rows.

    Score variants (AttnFuse, Table 6: sliding window W=256, causal + ALiBi),
    both on top of the causal mask.  Readings: ``window`` = W > 0 keeps key j
    for query i iff i - W < j <= i (the window counts the query's own key);
    ``alibi_slopes`` [Hq] adds slope_h * (j - i) to each score after the
    scaling (the linear-bias definition of ALiBi, a non-positive bias for
    visible keys).  Returns (o [B,Hq,R,Dv], lse [B,Hq,R]) as float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, _ = q.shape
    Hkv, Nk, Dv = k.shape[1], k.shape[2], v.shape[3]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    sel = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((B, Hq, len(sel), Dv))
    lse = np.full((B, Hq, len(sel)), NEG_INF)
    if Nk == 0 or len(sel) == 0:
        return o, lse
    for b in range(B):
        for h in range(Hq):
            kvh = h // group
            # pass 0: the score matrix, materialised in full
            s = (q[b, h, sel, :] @ k[b, kvh].T) * scale
            key_idx = np.arange(Nk)[None, :]
            if alibi_slopes is not None:
                s = s + float(_f64(alibi_slopes)[h]) * (key_idx - sel[:, None])
            if causal:
                s = np.where(key_idx <= sel[:, None], s, NEG_INF)
            if window:
                s = np.where(key_idx > sel[:, None] - window, s, NEG_INF)
            # level 1: row maximum
            m = s.max(axis=1)
            live = np.isfinite(m)
            m_safe = np.where(live, m, 0.0)
            # level 2: sum of exponentials relative to the maximum
            p = np.exp(s - m_safe[:, None])
            l = p.sum(axis=1)
            # level 3: exponential-weighted sum of V, then normalise
            acc = p @ v[b, kvh]
            with np.errstate(invalid="ignore", divide="ignore"):
                o[b, h] = np.where(live[:, None], acc / l[:, None], 0.0)
                lse[b, h] = np.where(live, m_safe + np.log(l), NEG_INF)
    return o, lse


def decode(q, k_cache, v_cache, scale):
    """Single-query attention over a KV cache (AttnFuse, Table 8, Q.N = 1).

    q is [B,Hq,D] or [B,Hq,1,D]; k_cache, v_cache are [B,Hkv,L,D].  No mask.
    This is the unsplit definition: splitting is an implementation choice whose
    result must equal this one.  Returns (o [B,Hq,D], lse [B,Hq]).
    """
    q = _f64(q)
    if q.ndim == 3:
        q = q[:, :, None, :]
    o, lse = attention(q, k_cache, v_cache, scale, causal=False)
    return o[:, :, 0, :], lse[:, :, 0]


def split_bounds(L, num_splits):
    """Key range [lo, hi) of each split.

    Reading (the FlashDecoding IR of RedFuser, Figure 13, did not survive
    extraction): contiguous chunks, split s covering
    [floor(s*L/S), floor((s+1)*L/S)).  Sizes differ by at most one; when
    L < S some splits are empty.
    """
    return [((s * L) // num_splits, ((s + 1) * L) // num_splits) for s in range(num_splits)]


def decode_partials(q, k_cache, v_cache, scale, num_splits):
    """Per-split partial results of decoding: the normalised O_s and lse_s of
    attention restricted to each split's keys (an empty split gives O_s = 0,
    lse_s = -inf).  Returns (o_part [B,Hq,S,D], lse_part [B,Hq,S])."""
    q, k, v = _f64(q), _f64(k_cache), _f64(v_cache)
    if q.ndim == 3:
        q = q[:, :, None, :]
    B, Hq, _, _ = q.shape
    L, Dv = k.shape[2], v.shape[3]
    o_part = np.zeros((B, Hq, num_splits, Dv))
    lse_part = np.full((B, Hq, num_splits), NEG_INF)
    for s, (lo, hi) in enumerate(split_bounds(L, num_splits)):
        o_s, lse_s = attention(q, k[:, :, lo:hi], v[:, :, lo:hi], scale, causal=False)
        o_part[:, :, s, :] = o_s[:, :, 0, :]
        lse_part[:, :, s] = lse_s[:, :, 0]
    return o_part, lse_part


def lse_merge(o_part, lse_part):
    """Combine partial attention results over disjoint key sets.

    o_part [..., S, D] holds normalised partial outputs, lse_part [..., S] their
    natural-log LSEs.  The combined result is LSE = ln sum_s exp(lse_s) and
    O = sum_s exp(lse_s - LSE) O_s: the level-2 sum and level-3 weighted sum of
    the whole key set rebuilt from the parts (reduce op + over the splits,
    combine op * for the rescale; RedFuser, Table 1).  The log-sum-exp is
    evaluated relative to the largest lse_s so that exp does not overflow.
    A row whose parts are all empty (every lse_s = -inf) gives O = 0,
    LSE = -inf.  Returns (o [..., D], lse [...]).
    """
    o_part, lse_part = _f64(o_part), _f64(lse_part)
    mx = lse_part.max(axis=-1)
    live = np.isfinite(mx)
    mx_safe = np.where(live, mx, 0.0)
    w = np.exp(lse_part - mx_safe[..., None])
    total = w.sum(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(live, mx_safe + np.log(total), NEG_INF)
        weight = np.where(live[..., None], np.exp(lse_part - np.where(live, lse, 0.0)[..., None]), 0.0)
    o = (weight[..., None] * o_part).sum(axis=-2)
    return o, lse


def layernorm(x, residual, gamma, beta, eps):
    """Residual add followed by LayerNorm over the last axis.

    "Operator Fusion", section 2, Pattern 2 lists the three passes: mean
    (reduction), variance about that mean (reduction), then
    (x - mean) / sqrt(var) * gamma + beta (element-wise); section 4's kernels
    add the residual first and place eps inside the square root.
    Reading: the variance is the biased one (divide by n), as in the section 4
    CUDA and Triton kernels.  Returns (y, h) with h = x + residual.
    """
    x, r, g, b = _f64(x), _f64(residual), _f64(gamma), _f64(beta)
    h = x + r                                              # element-wise prologue
    n = h.shape[-1]
    mean = h.sum(axis=-1, keepdims=True) / n               # pass 1
    var = ((h - mean) ** 2).sum(axis=-1, keepdims=True) / n  # pass 2 (biased)
    y = (h - mean) / np.sqrt(var + eps) * g + b            # pass 3
    return y, h


def rmsnorm(x, residual, gamma, eps):
    """Residual add followed by RMSNorm over the last axis.

    "Operator Fusion", section 3, lists RMSNorm beside LayerNorm as a fusible
    reduction + normalise pattern but prints no formula.  Reading (the usual
    definition): one reduction level, the mean of squares, then the element-wise
    level y = h / sqrt(mean(h^2) + eps) * gamma, with eps inside the root as in
    the guide's LayerNorm kernels and no bias.  Returns (y, h) with h = x + r.
    """
    x, r, g = _f64(x), _f64(residual), _f64(gamma)
    h = x + r
    n = h.shape[-1]
    ms = (h * h).sum(axis=-1, keepdims=True) / n          # the one reduction level
    y = h / np.sqrt(ms + eps) * g                          # element-wise level
    return y, h


def softmax_xent(logits, targets, ignore_index=-100):
    """Softmax cross-entropy per row, with its log-sum-exp and gradient.

    "Operator Fusion", section 3, lists softmax + cross-entropy (training loss)
    as a fusible pattern; it is a cascade of the same kind as attention's
    softmax: the row maximum m (level 1, reduce op max), l = sum_j exp(z_j - m)
    (level 2, reduce op +), then loss = m + ln l - z_target.  Readings: natural
    log; a row whose target equals ``ignore_index`` has loss 0 and gradient 0;
    the gradient is d loss / d z = softmax(z) - onehot(target), unscaled.
    Returns (loss [rows], lse [rows], grad [rows, V]) as float64.
    """
    z = _f64(logits)
    t = np.asarray(targets.detach().cpu().numpy() if hasattr(targets, "detach") else targets, dtype=np.int64)
    m = z.max(axis=-1, keepdims=True)                     # level 1
    l = np.exp(z - m).sum(axis=-1, keepdims=True)         # level 2
    lse = (m + np.log(l))[..., 0]
    valid = t != ignore_index
    tz = np.where(valid, z[np.arange(z.shape[0]), np.where(valid, t, 0)], 0.0)
    loss = np.where(valid, lse - tz, 0.0)
    grad = np.exp(z - lse[:, None])
    grad[np.arange(z.shape[0])[valid], t[valid]] -= 1.0
    grad[~valid] = 0.0
    return loss, lse, grad


def alibi_slopes(n_heads):
    """Head slopes of ALiBi (the linear-bias definition): the geometric sequence
    2^(-8 (h+1) / H) for h = 0..H-1.  The pages name ALiBi (AttnFuse, Table 6)
    without its slopes; this is the usual choice."""
    return np.array([2.0 ** (-8.0 * (h + 1) / n_heads) for h in range(n_heads)])


def rope(x, positions, base=10000.0):
    """Rotary position embedding of the rows of x.

    AttnFuse names RoPE as the pre-matmul transformation of Q and K used by
    every major LLM (Abstract; Figure 1) but prints no formula.  Reading (the
    usual definition, in the rotate-half pairing of the Llama models the page
    names): for head dimension D and i < D/2, the pair (x_i, x_{i+D/2}) of a
    row at position p is turned by the angle p * base^(-2i/D):
        y_i       = x_i cos(theta) - x_{i+D/2} sin(theta)
        y_{i+D/2} = x_i sin(theta) + x_{i+D/2} cos(theta)

    Shapes: x [..., N, D] with D even; positions [N] (integers).  Returns y as
    float64 with the shape of x.
    """
    x = _f64(x)
    D = x.shape[-1]
    if D % 2:
        raise ValueError("rope needs an even head dimension")
    half = D // 2
    pos = np.asarray(positions, dtype=np.float64).reshape(-1, 1)          # [N, 1]
    inv_freq = float(base) ** (-2.0 * np.arange(half, dtype=np.float64) / D)  # [D/2]
    theta = pos * inv_freq[None, :]                                         # [N, D/2]
    c, s = np.cos(theta), np.sin(theta)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)
