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


def test_merge_large_lse_values(rf):
    o_part, lse_part = inputs.merge_inputs(64, 16, 128, seed=3)
    lse_part = lse_part * 50 + 300  # exp(lse) alone would overflow fp32
    o, lse = run(rf, o_part, lse_part, torch.float32)
    ro, rl = oracle.lse_merge(o_part, lse_part)
    # fp32 floor: lse_s ~ 300 +- 200 is itself rounded to +-3e-5 absolute, so each
    # weight exp(lse_s - LSE) carries ~3e-5 relative error: allow 1e-4 here.
    rl2 = np.linalg.norm(o.numpy() - ro) / np.linalg.norm(ro)
    mr = np.abs(o.numpy() - ro).max() / np.abs(ro).max()
    assert rl2 <= 1e-5 and mr <= 1e-4, (rl2, mr)
    check_lse(lse, rl, tol=1e-5 * 1000)


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
