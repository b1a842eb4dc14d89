"""GPU parity of rf_layernorm_fused against the fp64 oracle (through the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check16_wide, check32, to64
from test_golden import dec

pytestmark = pytest.mark.gpu
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def run(rf, x, r, g, b, eps, want_rout=False):
    dev = "cuda"
    args = [t.to(dev) if t is not None else None for t in (x, r, g, b)]
    res = rf.layernorm(*args, eps=eps, want_residual_out=want_rout)
    torch.cuda.synchronize()
    return res


def check(dtype, y, ref, what):
    return check32(y, ref, what) if dtype == "f32" else check16(y, ref, what)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,cols", [(1, 8), (5, 64), (9, 256), (7, 520), (33, 1024), (4, 4096),
                                       (3, 4104), (2, 12288), (17, 2056)])
def test_layernorm_shapes(rf, dtype, rows, cols):
    if dtype == "f32" and cols % 4:
        pytest.skip("f32 needs cols % 4 == 0")
    x, r, g, b = inputs.ln_inputs(rows, cols, dtype, seed=rows * 7 + cols)
    y = run(rf, x, r, g, b, 1e-5)
    ref, _ = oracle.layernorm(x, r, g, b, 1e-5)
    check(dtype, y, ref, f"{dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype,cols", [("bf16", 32768), ("f16", 32768), ("f32", 16384)])
def test_layernorm_max_cols(rf, dtype, cols):
    x, r, g, b = inputs.ln_inputs(3, cols, dtype, seed=11)
    y = run(rf, x, r, g, b, 1e-5)
    ref, _ = oracle.layernorm(x, r, g, b, 1e-5)
    check(dtype, y, ref, f"{dtype} max cols")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_layernorm_optional_operands_and_residual_out(rf, dtype):
    x, r, g, b = inputs.ln_inputs(6, 768, dtype, seed=12)
    # no residual, no affine
    y = run(rf, x, None, None, None, 1e-5)
    ref, _ = oracle.layernorm(x, torch.zeros_like(x), torch.ones_like(g), torch.zeros_like(b), 1e-5)
    check(dtype, y, ref, "plain")
    # residual_out holds h = x + r rounded to the dtype
    y, h = run(rf, x, r, g, b, 1e-3, want_rout=True)
    ref, href = oracle.layernorm(x, r, g, b, 1e-3)
    check(dtype, y, ref, "with residual_out")
    href_rounded = torch.from_numpy(href).to(torch.float32).to(DT[dtype]).float().numpy()
    np.testing.assert_array_equal(to64(h), href_rounded)


def test_layernorm_constant_rows_give_beta(rf):
    x = torch.full((4, 512), 2.5, dtype=torch.bfloat16)
    r = torch.full((4, 512), -0.5, dtype=torch.bfloat16)
    _, _, g, b = inputs.ln_inputs(1, 512, "bf16", seed=13)
    y = run(rf, x, r, g, b, 1e-5)
    np.testing.assert_array_equal(to64(y), np.broadcast_to(to64(b), (4, 512)))


def test_layernorm_golden_fixture(rf):
    with open(os.path.join(os.path.dirname(__file__), "golden", "layernorm_small_oracle.json")) as f:
        g = json.load(f)
    t = {k: torch.from_numpy(dec(g[k]).astype(np.float32)).to(torch.bfloat16) for k in ("x", "r", "gamma", "beta")}
    y = run(rf, t["x"], t["r"], t["gamma"], t["beta"], g["eps"])
    check16(y, dec(g["y"]), "golden")


def test_layernorm_large_mean_offset(rf):
    # Rows with |mean| >> std: the one-pass running M2 must not cancel, and the
    # centred value must not carry the rounding of the mean (~3e-5 at 1000,
    # which is 3e-3 in units of sigma = 0.01).  The fp32 bound holds.
    x, r, g, b = inputs.ln_inputs(8, 4096, "f32", seed=14)
    x = x * 0.01 + 1000.0
    y = run(rf, x, r * 0.0, g, b, 1e-5)
    ref, _ = oracle.layernorm(x, r * 0.0, g, b, 1e-5)
    check32(y, ref, "large mean")


def _rows_with_first_vector(rows, cols, dtype, first, scale=1.0, seed=15):
    """Rows of N(0, scale^2) whose first 16-byte vector is replaced by `first`
    (the kernel's shift is that vector's mean)."""
    x, r, g, b = inputs.ln_inputs(rows, cols, "f32", seed=seed)
    x = x * scale
    e = 4 if dtype == "f32" else 8
    x[:, :e] = first
    x = x.to(DT[dtype])
    return x, torch.zeros_like(x), g.to(DT[dtype]), b.to(DT[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("first,scale,cols", [
    (1000.0, 0.01, 4096),   # an outlier first vector: the one-pass M2 would cancel
    (0.9, 1.0, 4096),       # shift 0.9 sigma from the mean: the one-pass branch at its limit
    (1.1, 1.0, 4096),       # 1.1 sigma: the re-centring branch
    (40.0, 1.0, 1024),      # one warp per row (several rows per CTA)
    (40.0, 1.0, 16384),     # 1024 threads per row
])
def test_layernorm_shift_far_from_mean(rf, dtype, first, scale, cols):
    x, r, g, b = _rows_with_first_vector(6, cols, dtype, first, scale)
    # mix rows that do and do not need the second reduction in one CTA
    x[1::2] = inputs.ln_inputs(3, cols, dtype, seed=16)[0]
    y = run(rf, x, r, g, b, 1e-5)
    ref, _ = oracle.layernorm(x, r, g, b, 1e-5)
    # the outlier's own output reaches ~64 * gamma: bf16 holds it to one ulp there
    if dtype == "f32":
        check32(y, ref, f"shift far from mean ({first}, {scale}, {cols})")
    else:
        check16_wide(y, ref, DT[dtype], f"shift far from mean ({first}, {scale}, {cols})")


@pytest.mark.slow
def test_layernorm_full_size_sampled(rf):
    w = inputs.WORKLOADS["layernorm_residual_bf16"]
    x, r, g, b = inputs.make(w)
    y = run(rf, x, r, g, b, w.dims["eps"]).cpu()
    rows = np.unique(np.concatenate([[0, 1, w.dims["rows"] - 1],
                                     np.random.default_rng(0).integers(0, w.dims["rows"], 254)]))
    ref, _ = oracle.layernorm(x[rows], r[rows], g, b, w.dims["eps"])
    check16(y[rows], ref, "full-size sampled rows")
    assert torch.isfinite(y.float()).all()


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,cols", [(1, 8), (7, 520), (33, 1024), (4, 4096), (3, 4104), (2, 16384)])
def test_rmsnorm_shapes(rf, dtype, rows, cols):
    x, r, g, _ = inputs.ln_inputs(rows, cols, dtype, seed=rows + 3 * cols)
    y = rf.rmsnorm(x.cuda(), r.cuda(), g.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    ref, _ = oracle.rmsnorm(x, r, g, 1e-5)
    check(dtype, y, ref, f"rms {dtype} {rows}x{cols}")


def test_rmsnorm_optional_operands_and_residual_out(rf):
    x, r, g, _ = inputs.ln_inputs(5, 2048, "bf16", seed=31)
    y = rf.rmsnorm(x.cuda(), None, None, eps=1e-6)
    torch.cuda.synchronize()
    ref, _ = oracle.rmsnorm(x, torch.zeros_like(x), torch.ones_like(g), 1e-6)
    check16(y, ref, "rms plain")
    y, h = rf.rmsnorm(x.cuda(), r.cuda(), g.cuda(), eps=1e-5, want_residual_out=True)
    torch.cuda.synchronize()
    ref, href = oracle.rmsnorm(x, r, g, 1e-5)
    check16(y, ref, "rms with residual_out")
    np.testing.assert_array_equal(to64(h), torch.from_numpy(href).float().to(torch.bfloat16).float().numpy())


@pytest.mark.slow
def test_rmsnorm_full_size_sampled(rf):
    w = inputs.WORKLOADS["rmsnorm_residual_bf16"]
    x, r, g = inputs.make(w)
    y = rf.rmsnorm(x.cuda(), r.cuda(), g.cuda(), eps=w.dims["eps"]).cpu()
    rows = np.unique(np.concatenate([[0, w.dims["rows"] - 1], np.random.default_rng(2).integers(0, w.dims["rows"], 126)]))
    ref, _ = oracle.rmsnorm(x[rows], r[rows], g, w.dims["eps"])
    check16(y[rows], ref, "rms full-size sampled rows")
