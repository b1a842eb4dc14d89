"""GPU parity of rf_attn_decode_splitkv against the fp64 oracle (through the C ABI).

The final output is checked against the unsplit oracle; the per-split partials
left in the workspace are checked against the oracle's contiguous-split
partials."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check_lse, rel_l2, to64
from test_golden import dec

pytestmark = pytest.mark.gpu


def run(rf, q, k, v, S, scale):
    B, Hq, D = q.shape[0], q.shape[1], q.shape[-1]
    ws = rf.decode_workspace(B, Hq, D, S)
    ws.fill_(0xFF)  # poison: every byte the kernel must write is overwritten
    o, lse = rf.decode(q.cuda(), k.cuda(), v.cuda(), S, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    op, lp = rf.decode_partials_view(ws, B, Hq, D, S)
    return o.cpu(), lse.cpu(), op.cpu(), lp.cpu()


def check_partials(op, lp, rop, rlp):
    assert (np.isneginf(to64(lp)) == np.isneginf(rlp)).all()
    fin = np.isfinite(rlp)
    assert np.abs(to64(lp)[fin] - rlp[fin]).max() <= 1e-3
    assert rel_l2(op, rop) <= 5e-3 and np.abs(to64(op) - rop).max() <= 2e-2
    assert (to64(op)[~fin] == 0).all()


@pytest.mark.parametrize("B,Hq,Hkv,L,D,S,dtype", [
    (1, 8, 1, 40, 128, 3, "bf16"),
    (2, 16, 2, 1000, 128, 16, "bf16"),
    (1, 4, 1, 100, 64, 7, "f16"),
    (3, 6, 6, 333, 128, 5, "bf16"),       # G = 1
    (1, 8, 1, 5, 128, 8, "bf16"),         # L < S: empty splits
    (1, 8, 8, 64, 64, 1, "f16"),          # one split
    (2, 24, 4, 4096, 128, 16, "f16"),     # G = 6
    (1, 8, 1, 2048 * 3 + 17, 128, 3, "bf16"),
])
def test_decode_shapes(rf, B, Hq, Hkv, L, D, S, dtype):
    q, k, v = inputs.decode_inputs(B, Hq, Hkv, L, D, dtype, seed=L + S)
    scale = float(np.float32(1 / np.sqrt(D)))
    o, lse, op, lp = run(rf, q, k, v, S, scale)
    ro, rl = oracle.decode(q, k, v, scale)
    check16(o, ro, "decode o")
    check_lse(lse, rl, what="decode lse")
    rop, rlp = oracle.decode_partials(q, k, v, scale, S)
    check_partials(op, lp, rop, rlp)


def test_decode_golden_fixture(rf):
    with open(os.path.join(os.path.dirname(__file__), "golden", "decode_small_oracle.json")) as f:
        g = json.load(f)
    q, k, v = (torch.from_numpy(dec(g[n]).astype(np.float32)).to(torch.bfloat16) for n in ("q", "k", "v"))
    o, lse, op, lp = run(rf, q, k, v, g["num_splits"], g["scale"])
    check16(o, dec(g["o"])[:, :, :], "golden o")
    check_lse(lse, dec(g["lse"]), what="golden lse")
    check_partials(op, lp, dec(g["o_part"]), dec(g["lse_part"]))


def test_decode_constant_values_and_one_hot(rf):
    B, Hq, Hkv, L, D = 1, 8, 1, 3000, 128
    q, k, v = inputs.decode_inputs(B, Hq, Hkv, L, D, "bf16", seed=5)
    row = v[0, 0, 17].clone()
    vc = row.expand(B, Hkv, L, D).contiguous()
    o, _, _, _ = run(rf, q, k, vc, 16, 0.088388)
    np.testing.assert_allclose(to64(o), np.broadcast_to(to64(row), o.shape), rtol=0, atol=8e-3)
    # one key dominates for every head: its V row comes back
    kk = k.clone()
    kk[0, 0, 1234] = (q[0, :, 0].float().mean(0) * 40).to(torch.bfloat16)
    qq = q.clone()
    qq[0, :, 0] = kk[0, 0, 1234]
    o, _, _, _ = run(rf, qq, kk, v, 16, 1.0)
    check16(o[0], np.broadcast_to(to64(v[0, 0, 1234]), (8, D)), "one-hot")


def test_workspace_partials_merge_to_output(rf):
    q, k, v = inputs.decode_inputs(2, 8, 1, 5000, 128, "bf16", seed=6)
    o, lse, op, lp = run(rf, q, k, v, 16, 0.088388)
    mo, ml = oracle.lse_merge(to64(op), to64(lp))
    check16(o, mo, "merge of the kernel's own partials")
    check_lse(lse, ml, tol=1e-4)


@pytest.mark.slow
def test_decode_full_size_sampled(rf):
    """batch 16, 64q/8kv heads, D=128, L=32768, 16 splits (seed 3): sampled groups vs oracle."""
    w = inputs.WORKLOADS["decode_splitkv_bf16"]
    d = w.dims
    q, k, v = inputs.make(w)
    scale = float(np.float32(1 / np.sqrt(d["D"])))
    o, lse, op, lp = run(rf, q, k, v, d["splits"], scale)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    G = d["Hq"] // d["Hkv"]
    for b, hk in [(0, 0), (7, 3), (15, 7), (9, 5)]:
        sl = slice(hk * G, (hk + 1) * G)
        ro, rl = oracle.decode(q[b:b + 1, sl], k[b:b + 1, hk:hk + 1], v[b:b + 1, hk:hk + 1], scale)
        check16(o[b:b + 1, sl], ro, f"group {b},{hk}")
        check_lse(lse[b:b + 1, sl], rl, what=f"group {b},{hk}")
