"""Algorithmic work of each operation: the bytes and flops the method must move
or compute, independent of how a kernel does it.  Used for roofline figures.

Byte counts are the compulsory HBM traffic of the fused single-loop form: every
input read once, every output written once ("Operator Fusion" guide, section 1:
a fused residual + LayerNorm reads x and the residual and writes the output,
2 reads + 1 write).  Flop counts follow the FlashAttention convention: 4*D
flops per visible (query, key) pair (two multiply-adds per element of Q K^T and
of P V); a causal mask counts half the square.
"""
from __future__ import annotations

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def attn_flops(B, Hq, Nq, Nk, D, causal, window=0):
    """A sliding window counts its visible pairs exactly: sum_i min(i + 1, window)."""
    if causal and window:
        w = min(window, Nq)
        pairs = w * (w + 1) / 2.0 + (Nq - w) * window
        return 4.0 * B * Hq * pairs * D
    full = 4.0 * B * Hq * Nq * Nk * D
    return full / 2.0 if causal else full


def attn_bytes(B, Hq, Hkv, Nq, Nk, D, dtype, with_lse=True):
    e = ELEM_BYTES[dtype]
    q = B * Hq * Nq * D * e
    kv = 2 * B * Hkv * Nk * D * e
    o = B * Hq * Nq * D * e
    lse = B * Hq * Nq * 4 if with_lse else 0
    return q + kv + o + lse


def decode_bytes(B, Hq, Hkv, L, D, dtype, with_lse=True):
    """K and V caches read once, q read once, O (and LSE) written once.  The
    fp32 split partials' round trip through the workspace is not credited."""
    return attn_bytes(B, Hq, Hkv, 1, L, D, dtype, with_lse)


def decode_flops(B, Hq, L, D):
    return attn_flops(B, Hq, 1, L, D, False)


def merge_bytes(rows, num_splits, D, out_dtype, with_lse=True):
    """Partials read once (fp32 O_s and lse_s), merged O (and LSE) written once."""
    return rows * num_splits * (D + 1) * 4 + rows * D * ELEM_BYTES[out_dtype] + (rows * 4 if with_lse else 0)


def layernorm_bytes(rows, cols, dtype, affine=True, residual_out=False):
    """x and residual read once, y written once (+ h if residual_out); gamma and
    beta read once per call."""
    e = ELEM_BYTES[dtype]
    t = rows * cols * e
    return 3 * t + (t if residual_out else 0) + (2 * cols * e if affine else 0)


def xent_bytes(rows, vocab, dtype, with_lse=True):
    """Logits read once, int64 targets read, fp32 loss (and LSE) written once."""
    return rows * vocab * ELEM_BYTES[dtype] + rows * 8 + rows * 4 + (rows * 4 if with_lse else 0)


def ablation_bytes(op, variant, rows, cols, dtype):
    """Compulsory HBM traffic of each ablation variant (RedFuser, Figure 7: a
    level that is not fused into the one before re-reads that level's input).

    op "layernorm" (cols = row length; t = one [rows, cols] tensor):
      0, 1  x and r read once, y written once: 3t (+ gamma, beta)
      2     statistics read x, r; normalise reads x, r again and writes y: 5t
            (+ the per-row (mean, rstd) written and read back)
      3     h = x + r written, read by the mean, variance and normalise
            kernels: 2t + t + t + t + 2t = 7t (+ per-row statistics)
    op "xent" (cols = vocab; T = the logits):
      0     T read once
      1     the row is read twice by one CTA: 2T through the memory system,
            of which the second pass may be served by L2
      2     the max and sum-of-exponentials kernels each read T: 2T
    The small per-row vectors (targets, loss, lse, statistics) are included.
    """
    e = ELEM_BYTES[dtype]
    if op == "layernorm":
        t = rows * cols * e
        aff = 2 * cols * e
        return {0: 3 * t, 1: 3 * t, 2: 5 * t + 16 * rows, 3: 7 * t + 24 * rows}[variant] + aff
    if op == "xent":
        T = rows * cols * e
        small = rows * 8 + rows * 8  # int64 targets; fp32 loss and lse
        return {0: T, 1: 2 * T, 2: 2 * T + rows * 16}[variant] + small
    raise ValueError(op)


def rope_bytes(B, Hq, Hkv, N, D, dtype):
    """Q and K read once and written once (out of place or in place alike)."""
    e = ELEM_BYTES[dtype]
    return 2 * B * (Hq + Hkv) * N * D * e
