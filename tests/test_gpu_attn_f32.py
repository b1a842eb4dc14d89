"""GPU parity of rf_attn_fwd's exact fp32 path against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check32, check_lse

pytestmark = pytest.mark.gpu


def run(rf, q, k, v, scale, causal):
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def test_tiny_workload(rf):
    """B=1 H=1 Nq=Nk=128 D=64, fp32 ~ N(0,1) from seed 0, scale 1/sqrt(64), no mask."""
    w = inputs.WORKLOADS["attn_tiny_f32"]
    q, k, v = inputs.make(w)
    o, lse = run(rf, q, k, v, 0.125, False)
    ro, rl = oracle.attention(q, k, v, 0.125, False)
    check32(o, ro, "tiny")
    check_lse(lse, rl, tol=1e-5 * max(1, np.abs(rl).max()))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,causal", [
    (1, 1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 1, 4, True),
    (2, 4, 2, 77, 77, 64, True),
    (1, 2, 2, 33, 150, 128, False),
    (1, 8, 1, 100, 100, 100, True),
    (3, 2, 1, 17, 5, 36, False),
    (1, 1, 1, 300, 300, 128, True),
    (1, 2, 1, 200, 333, 64, False),   # several 64-row blocks and 32-key tiles, both ragged
    (1, 1, 1, 129, 129, 32, True),    # one output group per lane, a one-row last block
    (1, 3, 3, 65, 300, 96, False),    # three output groups per lane
    (2, 2, 2, 64, 64, 64, True),      # exactly one block and two tiles
])
def test_shapes(rf, B, Hq, Hkv, Nq, Nk, D, causal):
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, Nq, Nk, D, "f32", seed=Nq + D)
    scale = float(np.float32(1 / np.sqrt(D)))
    o, lse = run(rf, q, k, v, scale, causal)
    ro, rl = oracle.attention(q, k, v, scale, causal)
    check32(o, ro, "shape")
    check_lse(lse, rl, tol=1e-5 * max(1, np.abs(rl).max()))


def test_constant_v_and_softmax_sum(rf):
    q, k, _ = inputs.attn_inputs(1, 1, 1, 40, 40, 64, "f32", seed=3)
    v = torch.ones(1, 1, 40, 64)
    o, _ = run(rf, q, k, v, 0.125, True)
    np.testing.assert_allclose(o.numpy(), 1.0, rtol=0, atol=2e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_full_workload_b1_h8_n2048(rf, causal):
    """The B=1 H=8 N=2048 D=64 workload the bench times (64 key tiles per 64-row
    block, split 32 / 32 between the two warp groups), every output against the
    oracle; causal too, where the two halves of a block's keys differ in length."""
    w = inputs.WORKLOADS["attn_f32_d64_n2048"]
    q, k, v = inputs.make(w)
    o, lse = run(rf, q, k, v, 0.125, causal)
    ro, rl = oracle.attention(q, k, v, 0.125, causal)
    check32(o, ro, f"B=1 H=8 N=2048 causal={causal}")
    check_lse(lse, rl, tol=1e-5 * max(1, np.abs(rl).max()))
