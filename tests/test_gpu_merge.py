"""GPU parity of rf_lse_merge against the fp64 oracle (through the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check32, check_lse
from test_golden import dec

pytestmark = pytest.mark.gpu


def run(rf, o_part, lse_part, dtype):
    rows, S, D = o_part.shape
    o = torch.empty(rows, D, dtype=dtype, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    rf.rf_lse_merge(o_part.cuda(), lse_part.cuda(), o, lse)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("rows,S,D", [(1, 1, 4), (5, 2, 64), (1024, 16, 128), (37, 33, 128), (9, 256, 8),
                                      (3, 7, 512), (300, 5, 100)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_shapes(rf, rows, S, D, dtype):
    o_part, lse_part = inputs.merge_inputs(rows, S, D, seed=rows + S + D, empty_frac=0.25)
    o, lse = run(rf, o_part, lse_part, dtype)
    ro, rl = oracle.lse_merge(o_part, lse_part)
    if dtype == torch.float32:
        check32(o, ro, "merge f32")
    else:
        check16(o, ro, "merge 16-bit")
    check_lse(lse, rl, tol=1e-5 * max(1.0, float(np.abs(rl[np.isfinite(rl)]).max(initial=0.0))))
    empty = np.isneginf(rl)
    assert empty.any() and (o.float().numpy()[empty] == 0).all()


@pytest.mark.parametrize("centre,spread", [(300.0, 50.0), (1000.0, 100.0), (1000.0, 0.25), (-800.0, 30.0)])
def test_merge_large_lse_values(rf, centre, spread):
    # exp(lse) alone would overflow (or underflow) fp32.  Each weight is formed
    # against the largest lse_s, an input value, so the rounding of the merged
    # LSE (of the order of ulp(LSE)) does not enter the weights: the fp32 bound
    # holds unchanged.
    o_part, lse_part = inputs.merge_inputs(64, 16, 128, seed=3)
    lse_part = lse_part * spread + centre
    o, lse = run(rf, o_part, lse_part, torch.float32)
    ro, rl = oracle.lse_merge(o_part, lse_part)
    check32(o, ro, f"merge f32 at lse ~ {centre}")
    # the merged LSE rounds once at its own magnitude: a few ulps of max |LSE|
    ulp = float(np.spacing(np.float32(np.abs(rl[np.isfinite(rl)]).max())))
    check_lse(lse, rl, tol=4 * ulp)


def test_merge_nan_part_marks_row_invalid(rf):
    # A split kernel that gave up after a bounded wait writes lse_s = NaN; the
    # merged row must then be NaN rather than a plausible value built from the
    # other parts.  The other rows are unaffected.
    o_part, lse_part = inputs.merge_inputs(6, 5, 32, seed=9)
    lse_part[2, 3] = float("nan")
    for dtype in (torch.float32, torch.bfloat16):
        o, lse = run(rf, o_part, lse_part, dtype)
        assert torch.isnan(o[2].float()).all() and torch.isnan(lse[2])
        keep = [0, 1, 3, 4, 5]
        ro, rl = oracle.lse_merge(o_part[keep], lse_part[keep])
        (check32 if dtype == torch.float32 else check16)(o[keep], ro, "rows without NaN")
        check_lse(lse[keep], rl, tol=1e-5 * 20)


def test_merge_golden_fixture(rf):
    with open(os.path.join(os.path.dirname(__file__), "golden", "merge_small_oracle.json")) as f:
        g = json.load(f)
    o_part = torch.from_numpy(dec(g["o_part"]).astype(np.float32))
    lse_part = torch.from_numpy(dec(g["lse_part"]).astype(np.float32))
    o, lse = run(rf, o_part, lse_part, torch.float32)
    check32(o, dec(g["o"]), "golden")
    check_lse(lse, dec(g["lse"]), tol=1e-5 * 20)


def test_merge_null_lse(rf):
    o_part, lse_part = inputs.merge_inputs(10, 4, 16, seed=4)
    o = torch.empty(10, 16, dtype=torch.float32, device="cuda")
    rf.rf_lse_merge(o_part.cuda(), lse_part.cuda(), o, None)
    torch.cuda.synchronize()
    check32(o.cpu(), oracle.lse_merge(o_part, lse_part)[0])
