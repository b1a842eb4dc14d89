"""GPU parity of the ablation variants (fusion at different levels, incremental
vs non-incremental; RedFuser, Figures 6-7) against the fp64 oracle.

Every variant computes the same LayerNorm / cross-entropy as the fused
kernels, so each is held to the same tolerances.  The unfused LayerNorm
(variant 3) materialises h = x + r in the input dtype between its kernels, as
an unfused framework does, so its oracle input is that rounded h (with a zero
residual): rounding h to bf16 moves each output by up to 2^-9 of |h - mean| *
rstd * gamma, about 3e-2 at the tails, beyond the 16-bit max-abs bound.
"""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check32, to64

pytestmark = pytest.mark.gpu


def ln_variant(rf, x, r, g, b, eps, variant):
    x, r, g, b = (t.cuda() for t in (x, r, g, b))
    out = torch.empty_like(x)
    ws = rf.ablation_workspace(0, variant, x.shape[0], x.shape[1], x.dtype)
    rf.rf_layernorm_ablation(x, r, g, b, out, variant, workspace=ws, eps=eps)
    torch.cuda.synchronize()
    return out.cpu()


def ln_reference(x, r, g, b, eps, variant):
    """The oracle's LayerNorm of the values the variant normalises."""
    if variant == 3 and x.dtype != torch.float32:
        h = (x.float() + r.float()).to(x.dtype)  # the materialised intermediate, rounded to nearest even
        return oracle.layernorm(h, torch.zeros_like(h), g, b, eps)[0]
    return oracle.layernorm(x, r, g, b, eps)[0]


def xent_variant(rf, logits, targets, variant):
    logits, targets = logits.cuda(), targets.cuda()
    rows, V = logits.shape
    loss = torch.empty(rows, dtype=torch.float32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    ws = rf.ablation_workspace(1, variant, rows, V, logits.dtype)
    rf.rf_softmax_xent_ablation(logits, targets, loss, lse, variant, workspace=ws)
    torch.cuda.synchronize()
    return loss.cpu(), lse.cpu()


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,cols", [(1, 8), (5, 64), (7, 520), (33, 1024), (3, 4104), (2, 12288)])
def test_layernorm_variants(rf, variant, dtype, rows, cols):
    x, r, g, b = inputs.ln_inputs(rows, cols, dtype, seed=rows * 13 + cols)
    y = ln_variant(rf, x, r, g, b, 1e-5, variant)
    ref = ln_reference(x, r, g, b, 1e-5, variant)
    (check32 if dtype == "f32" else check16)(y, ref, f"LN variant {variant} {dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_layernorm_smem_variant_at_its_largest_row(rf, dtype):
    """Variant 1 holds the whole row on chip: 56,832 fp32 values fill 222 KiB."""
    x, r, g, b = inputs.ln_inputs(3, 56832, dtype, seed=21)
    y = ln_variant(rf, x, r, g, b, 1e-5, 1)
    ref, _ = oracle.layernorm(x, r, g, b, 1e-5)
    (check32 if dtype == "f32" else check16)(y, ref, "LN variant 1, 56832 columns")


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_layernorm_variants_large_mean(rf, variant):
    """A row mean far from zero: the two-pass and pairwise forms stay accurate."""
    x, r, g, b = inputs.ln_inputs(8, 4096, "f32", seed=22)
    x = x + 1000.0
    y = ln_variant(rf, x, r, g, b, 1e-5, variant)
    ref, _ = oracle.layernorm(x, r, g, b, 1e-5)
    assert np.abs(to64(y) - ref).max() <= 5e-3


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,V", [(1, 8), (7, 1000), (33, 32000), (5, 128256), (300, 4096)])
def test_xent_variants(rf, variant, dtype, rows, V):
    logits, targets = inputs.xent_inputs(rows, V, dtype, seed=rows * 3 + V)
    targets[::4] = -100
    loss, lse = xent_variant(rf, logits, targets, variant)
    rloss, rlse, _ = oracle.softmax_xent(logits, targets)
    tol = 1e-5 * max(1.0, float(np.abs(rlse).max())) if dtype == "f32" else 1e-3
    assert np.abs(to64(lse) - rlse).max() <= tol
    assert np.abs(to64(loss) - rloss).max() <= tol
    assert (to64(loss)[::4] == 0).all()


@pytest.mark.parametrize("variant", [1, 2])
def test_xent_variants_out_of_range_target(rf, variant):
    logits, targets = inputs.xent_inputs(4, 256, "bf16", seed=23)
    targets[1] = 256
    targets[2] = -7
    loss, lse = xent_variant(rf, logits, targets, variant)
    assert np.isnan(to64(loss)[[1, 2]]).all() and np.isfinite(to64(loss)[[0, 3]]).all()
    assert np.isfinite(to64(lse)).all()


@pytest.mark.slow
@pytest.mark.parametrize("variant", [1, 2, 3])
def test_layernorm_variants_full_size_sampled(rf, variant):
    w = inputs.WORKLOADS["layernorm_residual_bf16"]
    x, r, g, b = inputs.make(w)
    y = ln_variant(rf, x, r, g, b, w.dims["eps"], variant)
    rows = np.unique(np.concatenate([[0, w.dims["rows"] - 1],
                                     np.random.default_rng(variant).integers(0, w.dims["rows"], 126)]))
    ref = ln_reference(x[rows], r[rows], g, b, w.dims["eps"], variant)
    check16(y[rows], ref, f"LN variant {variant} full-size sampled rows")


@pytest.mark.slow
@pytest.mark.parametrize("variant", [1, 2])
def test_xent_variants_full_size_sampled(rf, variant):
    w = inputs.WORKLOADS["softmax_xent_bf16"]
    logits, targets = inputs.make(w)
    loss, lse = xent_variant(rf, logits, targets, variant)
    rows = np.unique(np.concatenate([[0, w.dims["rows"] - 1],
                                     np.random.default_rng(variant).integers(0, w.dims["rows"], 62)]))
    rloss, rlse, _ = oracle.softmax_xent(logits[rows], targets[rows])
    assert np.abs(to64(lse)[rows] - rlse).max() <= 1e-3
    assert np.abs(to64(loss)[rows] - rloss).max() <= 1e-3
