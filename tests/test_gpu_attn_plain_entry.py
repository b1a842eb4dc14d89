"""GPU parity of the plain rf_attn_fwd entry point (no options, no workspace)
against the fp64 oracle, through the C ABI: every dtype and path it serves."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check32, check_lse

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rf_attn_fwd_plain(rf, dtype, D, causal):
    B, Hq, Hkv, N = 1, 4, 2, 333  # GQA, a ragged last tile
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, N, N, D, dtype, seed=50 + D + int(causal))
    scale = float(np.float32(1 / np.sqrt(D)))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    rf.rf_attn_fwd(qd, kd, vd, o, lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, scale, causal)
    if dtype == "f32":
        check32(o.cpu(), ro, f"rf_attn_fwd f32 D={D} causal={causal}")
        check_lse(lse.cpu(), rl, tol=1e-5 * max(1.0, float(np.abs(rl).max())))
    else:
        check16(o.cpu(), ro, f"rf_attn_fwd {dtype} D={D} causal={causal}")
        check_lse(lse.cpu(), rl)


def test_rf_attn_fwd_plain_without_lse(rf):
    q, k, v = inputs.attn_inputs(2, 2, 2, 256, 256, 64, "f16", seed=57)
    o = torch.empty_like(q.cuda())
    rf.rf_attn_fwd(q.cuda(), k.cuda(), v.cuda(), o, None, scale=0.125)
    torch.cuda.synchronize()
    check16(o.cpu(), oracle.attention(q, k, v, 0.125, False)[0], "rf_attn_fwd, lse = NULL")
