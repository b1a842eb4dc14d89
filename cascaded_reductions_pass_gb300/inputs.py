"""Seeded synthetic inputs for the fused cascaded-reduction kernels.

This module only draws random numbers; it holds none of the arithmetic of
attention, decoding, the log-sum-exp merge or LayerNorm.  It is the one
module that both the oracle-based tests and the CUDA path consume, so that
both sides see bit-identical inputs.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws float32 values in argument order, and each tensor
is then cast to its target dtype with round-to-nearest-even.  Standard
normals come from ``torch.randn``; uniforms from ``torch.rand``.
"""
from __future__ import annotations

import dataclasses

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def _normal(g, shape, dtype, std=1.0):
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(dtype)


def attn_inputs(B, Hq, Hkv, Nq, Nk, D, dtype, seed):
    """q [B,Hq,Nq,D], k and v [B,Hkv,Nk,D], all ~ N(0,1) (drawn q, k, v)."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = _gen(seed)
    q = _normal(g, (B, Hq, Nq, D), dt)
    k = _normal(g, (B, Hkv, Nk, D), dt)
    v = _normal(g, (B, Hkv, Nk, D), dt)
    return q, k, v


def decode_inputs(B, Hq, Hkv, L, D, dtype, seed):
    """q [B,Hq,1,D], k_cache and v_cache [B,Hkv,L,D], all ~ N(0,1)."""
    return attn_inputs(B, Hq, Hkv, 1, L, D, dtype, seed)


def ln_inputs(rows, cols, dtype, seed):
    """x, r [rows,cols] ~ N(0,1); gamma [cols] ~ U(0.5,1.5); beta [cols] ~ N(0, 0.1^2)."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = _gen(seed)
    x = _normal(g, (rows, cols), dt)
    r = _normal(g, (rows, cols), dt)
    gamma = (torch.rand(cols, generator=g, dtype=torch.float32) + 0.5).to(dt)
    beta = _normal(g, (cols,), dt, std=0.1)
    return x, r, gamma, beta


def xent_inputs(rows, vocab, dtype, seed, scale=2.0):
    """logits [rows,vocab] ~ N(0, scale^2); targets [rows] int64 uniform in [0, vocab)."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    g = _gen(seed)
    logits = _normal(g, (rows, vocab), dt, std=scale)
    targets = torch.randint(0, vocab, (rows,), generator=g, dtype=torch.int64)
    return logits, targets


def merge_inputs(rows, num_splits, D, seed, empty_frac=0.0):
    """Arbitrary split partials: o_part [rows,S,D] ~ N(0,1), lse_part [rows,S] ~ 4*N(0,1).

    With ``empty_frac`` > 0 that fraction of the (row, split) slots gets
    lse = -inf and o = 0 (an empty split); every eighth row is made fully empty.
    """
    g = _gen(seed)
    o = torch.randn(rows, num_splits, D, generator=g, dtype=torch.float32)
    lse = torch.randn(rows, num_splits, generator=g, dtype=torch.float32) * 4.0
    if empty_frac > 0.0:
        mask = torch.rand(rows, num_splits, generator=g) < empty_frac
        mask[::8, :] = True
        lse[mask] = float("-inf")
        o[mask] = 0.0
    return o, lse


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: the sizes, dtype and seed of one benchmark case."""

    name: str
    kind: str  # "attn" | "decode" | "layernorm"
    dtype: str
    seed: int
    dims: dict

    def describe(self) -> str:
        d = ",".join(f"{k}={v}" for k, v in self.dims.items())
        return f"{self.name}({d},{self.dtype},seed={self.seed})"


# The five synthetic workloads: a tiny fp32 attention, a non-causal fp16
# attention (B=4 H=12 N=4096 D=64), a causal GQA bf16 attention (B=2 Hq=32
# Hkv=8 N=8192 D=128), a split-KV decode on the Llama-3-70B head geometry
# (batch 16, 64q/8kv heads, D=128, 32768 cached keys, 16 splits) and a
# residual+LayerNorm over 16384 x 4096; and a residual+RMSNorm of the same
# shape and a softmax cross-entropy over 4096 rows of a 128256-entry
# vocabulary (the Llama-3 vocabulary size), the next workloads after the hot
# path.
WORKLOADS = {
    "attn_tiny_f32": Workload("attn_tiny_f32", "attn", "f32", 0,
                              dict(B=1, Hq=1, Hkv=1, N=128, D=64, causal=0)),
    "attn_fwd_f16_d64": Workload("attn_fwd_f16_d64", "attn", "f16", 1,
                                 dict(B=4, Hq=12, Hkv=12, N=4096, D=64, causal=0)),
    "attn_fwd_causal_gqa_bf16_d128": Workload(
        "attn_fwd_causal_gqa_bf16_d128", "attn", "bf16", 2,
        dict(B=2, Hq=32, Hkv=8, N=8192, D=128, causal=1)),
    "decode_splitkv_bf16": Workload("decode_splitkv_bf16", "decode", "bf16", 3,
                                    dict(B=16, Hq=64, Hkv=8, L=32768, D=128, splits=16)),
    "layernorm_residual_bf16": Workload("layernorm_residual_bf16", "layernorm", "bf16", 4,
                                        dict(rows=16384, cols=4096, eps=1e-5)),
    "rmsnorm_residual_bf16": Workload("rmsnorm_residual_bf16", "rmsnorm", "bf16", 6,
                                      dict(rows=16384, cols=4096, eps=1e-5)),
    "softmax_xent_bf16": Workload("softmax_xent_bf16", "xent", "bf16", 7,
                                  dict(rows=4096, vocab=128256)),
    # the score variants of AttnFuse's Table 6 on the non-causal workload's shape
    "attn_sw256_f16_d64": Workload("attn_sw256_f16_d64", "attn", "f16", 8,
                                   dict(B=4, Hq=12, Hkv=12, N=4096, D=64, causal=1, window=256)),
    "attn_causal_alibi_f16_d64": Workload("attn_causal_alibi_f16_d64", "attn", "f16", 9,
                                          dict(B=4, Hq=12, Hkv=12, N=4096, D=64, causal=1, alibi=1)),
    # the exact fp32 path at a size where its FFMA throughput, not launch latency, decides
    "attn_f32_d64_n2048": Workload("attn_f32_d64_n2048", "attn", "f32", 11,
                                   dict(B=1, Hq=8, Hkv=8, N=2048, D=64, causal=0)),
    # rotary embedding of Q and K at AttnFuse's RoPE + causal shape (Tables 4-5)
    "rope_qk_f16_d64": Workload("rope_qk_f16_d64", "rope", "f16", 10,
                                dict(B=4, Hq=12, Hkv=12, N=4096, D=64, base=10000.0)),
}


def make(workload: Workload):
    """Draw the inputs of one workload (CPU tensors, target dtype)."""
    d = workload.dims
    if workload.kind == "attn":
        return attn_inputs(d["B"], d["Hq"], d["Hkv"], d["N"], d["N"], d["D"],
                           workload.dtype, workload.seed)
    if workload.kind == "decode":
        return decode_inputs(d["B"], d["Hq"], d["Hkv"], d["L"], d["D"],
                             workload.dtype, workload.seed)
    if workload.kind == "layernorm":
        return ln_inputs(d["rows"], d["cols"], workload.dtype, workload.seed)
    if workload.kind == "rmsnorm":
        x, r, g, _ = ln_inputs(d["rows"], d["cols"], workload.dtype, workload.seed)
        return x, r, g
    if workload.kind == "xent":
        return xent_inputs(d["rows"], d["vocab"], workload.dtype, workload.seed)
    if workload.kind == "rope":
        q, k, _ = attn_inputs(d["B"], d["Hq"], d["Hkv"], d["N"], d["N"], d["D"], workload.dtype, workload.seed)
        return q, k
    raise ValueError(workload.kind)
