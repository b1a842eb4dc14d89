"""GPU parity of rf_rope_qk (rotary position embedding of Q and K) against the
fp64 oracle, and of rotary attention (RoPE pass, then the attention kernel)
against the oracle's attention of the oracle's rotated inputs."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check_lse, rel_l2, to64

pytestmark = pytest.mark.gpu


def run(rf, q, k, base, pos_offset, in_place):
    qd, kd = q.cuda(), (k.cuda() if k is not None else None)
    if in_place:
        rf.rf_rope_qk(qd, kd, base=base, pos_offset=pos_offset)
        qo, ko = qd, kd
    else:
        qo = torch.empty_like(qd)
        ko = torch.empty_like(kd) if kd is not None else None
        rf.rf_rope_qk(qd, kd, qo, ko, base=base, pos_offset=pos_offset)
    torch.cuda.synchronize()
    return qo.cpu(), (ko.cpu() if ko is not None else None)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B,Hq,Hkv,N,D,base,off", [
    (1, 1, 1, 1, 64, 10000.0, 0),
    (1, 2, 1, 7, 64, 10000.0, 0),        # fewer positions than one CTA's block
    (2, 4, 2, 300, 128, 500000.0, 0),    # GQA, ragged N
    (1, 3, 3, 65, 256, 10000.0, 12345),
    (2, 2, 1, 1000, 64, 10000.0, 1000000),  # large positions: angles in the millions of radians
])
def test_rope_shapes(rf, dtype, B, Hq, Hkv, N, D, base, off):
    q, k, _ = inputs.attn_inputs(B, Hq, Hkv, N, N, D, dtype, seed=N + D + off % 97)
    pos = np.arange(off, off + N)
    for in_place in (False, True):
        qo, ko = run(rf, q, k, base, off, in_place)
        rq, rk = oracle.rope(q, pos, base), oracle.rope(k, pos, base)
        check16(qo, rq, f"q {dtype} in_place={in_place}")
        check16(ko, rk, f"k {dtype} in_place={in_place}")
        # only the final 16-bit rounding separates the two: half an ulp, relative
        bound = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
        assert rel_l2(qo, rq) <= bound and rel_l2(ko, rk) <= bound


def test_rope_q_only(rf):
    q, _, _ = inputs.attn_inputs(1, 4, 4, 129, 129, 64, "bf16", seed=3)
    qo, ko = run(rf, q, None, 10000.0, 5, False)
    assert ko is None
    check16(qo, oracle.rope(q, np.arange(5, 134)), "q only")


def test_rope_then_attention_matches_oracle(rf):
    """Rotary causal attention: RoPE pass, then the tensor-core attention kernel."""
    B, H, N, D = 1, 4, 1000, 64
    q, k, v = inputs.attn_inputs(B, H, H, N, N, D, "f16", seed=11)
    scale = float(np.float32(1 / np.sqrt(D)))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rf.rf_rope_qk(qd, kd)
    o, lse = rf.attention(qd, kd, vd, scale=scale, causal=True)
    torch.cuda.synchronize()
    pos = np.arange(N)
    ro, rl = oracle.attention(oracle.rope(q, pos), oracle.rope(k, pos), v, scale, True)
    check16(o.cpu(), ro, "rope + causal attention")
    check_lse(lse.cpu(), rl, what="rope + causal attention lse")


@pytest.mark.slow
def test_rope_workload_sampled(rf):
    w = inputs.WORKLOADS["rope_qk_f16_d64"]
    q, k = inputs.make(w)
    d = w.dims
    qo, ko = run(rf, q, k, d["base"], 0, False)
    rows = np.random.default_rng(0).integers(0, d["N"], 64)
    pos = np.arange(d["N"])
    for b, h in ((0, 0), (d["B"] - 1, d["Hq"] - 1)):
        check16(qo[b, h, rows], oracle.rope(q[b:b + 1, h:h + 1], pos, d["base"])[0, 0, rows], "q sampled")
        check16(ko[b, h, rows], oracle.rope(k[b:b + 1, h:h + 1], pos, d["base"])[0, 0, rows], "k sampled")
