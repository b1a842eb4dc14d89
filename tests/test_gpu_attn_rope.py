"""GPU parity of attention with the rotary embedding applied inside the kernel
(rf_attn_fwd_ex, rope = 1: Q rows; rope = 2: Q and K rows) against the fp64
oracle's attention of the oracle's rotated rows, through the C ABI.

With rope = 1 the kernel turns Q with the same angle function as the separate
pass (rf_rope_qk), so attention over K rotated by that pass must equal, bit for
bit, the separate pass followed by plain attention."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16

pytestmark = pytest.mark.gpu


def check_lse_rotated(lse, ref, q, k, scale, dtype):
    """LSE of attention over rows rotated on the GPU.  The kernel rounds its
    fp32 rotation to the 16-bit format; where that value lies within the
    rotation's own error (~1e-6) of a rounding boundary it can land one ulp
    (2^-7 relative for bf16, 2^-10 for f16) from the oracle's correctly rounded
    row.  One such element moves a score by at most scale * ulp * |q_i| |k_i|,
    and the LSE by no more than its largest score change.  So: at most 1% of
    rows beyond the 16-bit LSE tolerance of 1e-3, none beyond that bound."""
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref)
    u = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
    qm, km = float(q.float().abs().max()), float(k.float().abs().max())
    bound = 1e-3 + 2 * scale * u * qm * km
    assert (err > 1e-3).mean() <= 0.01 and err.max() <= bound, (float(err.max()), float((err > 1e-3).mean()), bound)


def oracle_rope_attention(q, k, v, scale, causal, base, off, window=0):
    """The oracle's rotation of Q and K, rounded to the inputs' dtype (the
    tensor core reads the rotated rows in that format, as it reads the rows the
    separate pass writes), then the oracle's attention."""
    pos_q = np.arange(q.shape[2]) + off
    pos_k = np.arange(k.shape[2]) + off
    rq = torch.from_numpy(oracle.rope(q, pos_q, base)).to(q.dtype)
    rk = torch.from_numpy(oracle.rope(k, pos_k, base)).to(k.dtype)
    return oracle.attention(rq, rk, v, scale, causal, window=window)


@pytest.mark.parametrize("rope", [1, 2])
@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,dtype,window,off", [
    (1, 2, 1, 333, 64, False, "f16", 0, 0),        # GQA, ragged last tile, split tail
    (1, 2, 2, 256, 128, False, "bf16", 0, 0),
    (2, 4, 2, 384, 64, True, "bf16", 0, 7),        # causal, 1.5 CTA tiles, position offset
    (1, 2, 1, 640, 128, True, "f16", 0, 0),
    (1, 3, 3, 700, 64, True, "f16", 256, 0),       # sliding window (per-unit kernel)
    (1, 2, 1, 300, 128, True, "bf16", 100, 40000),  # large positions
    (1, 1, 1, 1, 64, False, "f16", 0, 5),
    (1, 4, 4, 1024, 64, False, "bf16", 0, 0),
])
def test_fused_rope_matches_oracle(rf, rope, B, Hq, Hkv, N, D, causal, dtype, window, off):
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, N, N, D, dtype, seed=N + D + rope)
    scale = float(np.float32(1 / np.sqrt(D)))
    pos = np.arange(N) + off
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if rope == 1:  # K arrives already rotated (as from a cache written by the separate pass)
        kd = kd.clone()
        rf.rf_rope_qk(kd, base=10000.0, pos_offset=off)
    q0, k0 = qd.clone(), kd.clone()
    o, lse = rf.attention(qd, kd, vd, scale=scale, causal=causal, window=window, rope=rope, rope_pos_offset=off)
    torch.cuda.synchronize()
    assert torch.equal(qd, q0) and torch.equal(kd, k0), "inputs must not be modified"
    ro, rl = oracle_rope_attention(q, k, v, scale, causal, 10000.0, off, window)
    check16(o.cpu(), ro, f"rope={rope} {dtype} D={D} causal={causal} W={window}")
    check_lse_rotated(lse, rl, q, k, scale, dtype)


@pytest.mark.parametrize("dtype,D,causal", [("f16", 64, False), ("bf16", 128, True), ("f16", 128, False),
                                            ("bf16", 64, True)])
def test_fused_q_rotation_equals_separate_pass_bitwise(rf, dtype, D, causal):
    B, Hq, Hkv, N = 1, 4, 2, 520
    q, k, v = (t.cuda() for t in inputs.attn_inputs(B, Hq, Hkv, N, N, D, dtype, seed=77 + D))
    scale = float(np.float32(1 / np.sqrt(D)))
    qr, kr = q.clone(), k.clone()
    rf.rf_rope_qk(qr, kr, base=500000.0, pos_offset=3)
    o_sep, lse_sep = rf.attention(qr, kr, v, scale=scale, causal=causal)
    o_fused, lse_fused = rf.attention(q, kr, v, scale=scale, causal=causal, rope=1, rope_base=500000.0,
                                      rope_pos_offset=3)
    torch.cuda.synchronize()
    assert torch.equal(o_sep, o_fused) and torch.equal(lse_sep, lse_fused)


def test_fused_qk_rotation_close_to_separate_pass(rf):
    # K turned inside the kernel uses angle-sum products for its cosines and
    # sines: equal to the separate pass up to the rounding of those values.
    q, k, v = (t.cuda() for t in inputs.attn_inputs(2, 4, 2, 777, 777, 64, "f16", seed=81))
    qr, kr = q.clone(), k.clone()
    rf.rf_rope_qk(qr, kr)
    o_sep, lse_sep = rf.attention(qr, kr, v, scale=0.125)
    o_fused, lse_fused = rf.attention(q, k, v, scale=0.125, rope=2)
    torch.cuda.synchronize()
    assert (o_sep.float() - o_fused.float()).abs().max().item() <= 4e-3
    assert (lse_sep - lse_fused).abs().max().item() <= 1e-3
