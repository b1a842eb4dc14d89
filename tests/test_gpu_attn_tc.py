"""GPU parity of rf_attn_fwd's tcgen05 path (fp16/bf16, D in {64, 128}) against the
fp64 oracle, through the C ABI.  Small and ragged shapes are compared element by
element; the two full-size workloads on sampled query rows."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check_lse, to64
from test_golden import dec

pytestmark = pytest.mark.gpu


def run(rf, q, k, v, scale, causal):
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,causal,dtype", [
    (1, 1, 1, 128, 128, 64, False, "f16"),
    (1, 1, 1, 128, 128, 128, False, "bf16"),
    (1, 2, 1, 256, 256, 64, True, "f16"),
    (1, 2, 2, 200, 200, 128, False, "bf16"),   # ragged tiles
    (2, 4, 2, 384, 384, 128, True, "bf16"),    # GQA, causal, 1.5 CTA tiles
    (1, 1, 1, 1, 1, 64, False, "f16"),
    (1, 1, 1, 1, 1, 128, True, "bf16"),
    (1, 3, 1, 1000, 1000, 64, True, "bf16"),
    (1, 2, 1, 64, 64, 128, True, "f16"),
    (1, 2, 2, 100, 700, 64, False, "f16"),     # Nq != Nk
    (1, 2, 1, 513, 300, 128, False, "f16"),
    (1, 4, 4, 1024, 1024, 64, False, "bf16"),
    (1, 8, 2, 640, 640, 128, True, "f16"),
])
def test_shapes(rf, B, Hq, Hkv, Nq, Nk, D, causal, dtype):
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, Nq, Nk, D, dtype, seed=Nq + Nk + D)
    scale = float(np.float32(1 / np.sqrt(D)))
    o, lse = run(rf, q, k, v, scale, causal)
    ro, rl = oracle.attention(q, k, v, scale, causal)
    check16(o, ro, f"{dtype} D={D} causal={causal}")
    check_lse(lse, rl, what="lse")


def test_golden_fixture(rf):
    with open(os.path.join(os.path.dirname(__file__), "golden", "attn_small_oracle.json")) as f:
        g = json.load(f)
    q, k, v = (torch.from_numpy(dec(g[n]).astype(np.float32)).to(torch.float16) for n in ("q", "k", "v"))
    for causal in (0, 1):
        o, lse = run(rf, q, k, v, g["scale"], bool(causal))
        check16(o, dec(g[f"o_causal{causal}"]), f"golden causal={causal}")
        check_lse(lse, dec(g[f"lse_causal{causal}"]), what="golden lse")


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(rf, causal):
    # V = identity (Nk = D = 64): each output row is the softmax row itself.
    q, k, _ = inputs.attn_inputs(1, 2, 2, 64, 64, 64, "bf16", seed=40)
    v = torch.eye(64, dtype=torch.bfloat16).expand(1, 2, 64, 64).contiguous()
    o, _ = run(rf, q * 3, k, v, 0.125, causal)
    s = to64(o).sum(-1)
    assert np.abs(s - 1).max() <= 2e-2
    if causal:
        assert (np.triu(to64(o)[0, 0], 1) == 0).all()


def test_constant_v_and_large_scores(rf):
    q, k, _ = inputs.attn_inputs(1, 2, 1, 500, 500, 128, "f16", seed=41)
    row = torch.randn(128).to(torch.float16)
    v = row.expand(1, 1, 500, 128).contiguous()
    o, _ = run(rf, q * 4, k * 4, v, 1.0, True)  # scores of several hundred: exp must not overflow
    assert np.abs(to64(o) - to64(row)).max() <= 2e-2


def test_one_hot_dominant_key(rf):
    q, k, v = inputs.attn_inputs(1, 1, 1, 256, 256, 64, "bf16", seed=42)
    targets = torch.randperm(256, generator=torch.Generator().manual_seed(0))
    q2 = (k[0, 0, targets].float() * 8).to(torch.bfloat16)[None, None]
    o, _ = run(rf, q2, k, v, 1.0, False)
    check16(o[0, 0], to64(v[0, 0, targets]), "one-hot")


# Scores that climb from key tile to key tile, so that a row's running max is
# overtaken in every way the kernel handles it: on the row's first tile, in the
# first half (keys 0-63) of a later tile, in its second half only, and not at
# all.  Levels are natural-log units per half tile of 64 keys; a jump of 14 is
# 2^20 in P.  In the first pattern the running max is first overtaken in a
# second half, in the second pattern in a first half.
RISING_LEVELS = {"second_half_first": [[0, 0], [0, 14], [30, 30], [31, 29], [5, 60]],
                 "first_half_first": [[0, 0], [1, 0], [20, 20], [20, 21], [40, 40]]}


@pytest.mark.parametrize("D,dtype,causal,window,alibi,levels", [
    (64, "f16", False, 0, False, "second_half_first"),
    (64, "bf16", False, 0, False, "first_half_first"),
    (64, "bf16", True, 0, False, "second_half_first"),
    (128, "f16", True, 0, False, "first_half_first"),
    (128, "bf16", False, 0, False, "second_half_first"),
    (64, "f16", True, 300, True, "second_half_first"),
])
def test_rising_scores_take_every_rescale_path(rf, D, dtype, causal, window, alibi, levels):
    pattern = RISING_LEVELS[levels]
    N, H = 128 * len(pattern), 2
    rng = np.random.default_rng(D + window)
    u = rng.standard_normal(D)
    u /= np.linalg.norm(u)
    level = np.repeat(np.asarray(pattern, dtype=np.float64).reshape(-1), 64)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    q = (np.sqrt(D) * u + 0.05 * rng.standard_normal((1, H, N, D)))
    k = level[:, None] * u + 0.3 * rng.standard_normal((1, H, N, D))
    v = rng.standard_normal((1, H, N, D))
    q, k, v = (torch.from_numpy(x).to(tdt) for x in (q, k, v))
    scale = float(np.float32(1 / np.sqrt(D)))
    slopes = oracle.alibi_slopes(H) if alibi else None
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, window=window,
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda() if alibi else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, scale, causal, window=window, alibi_slopes=slopes)
    check16(o.cpu(), ro, f"rising scores D={D} causal={causal} W={window}")
    check_lse(lse.cpu(), rl, what="rising scores lse")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["attn_fwd_f16_d64", "attn_fwd_causal_gqa_bf16_d128"])
def test_full_size_sampled(rf, name):
    w = inputs.WORKLOADS[name]
    d = w.dims
    q, k, v = inputs.make(w)
    scale = float(np.float32(1 / np.sqrt(d["D"])))
    o, lse = run(rf, q, k, v, scale, bool(d["causal"]))
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, d["N"] - 1], rng.integers(0, d["N"], 57)]))
    G = d["Hq"] // d["Hkv"]
    for b, h in [(0, 0), (d["B"] - 1, d["Hq"] - 1), (0, d["Hq"] // 2 + 1)]:
        kv = h // G
        ro, rl = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, kv:kv + 1], v[b:b + 1, kv:kv + 1], scale,
                                  bool(d["causal"]), rows=rows)
        check16(o[b:b + 1, h:h + 1, rows], ro, f"{name} b={b} h={h}")
        check_lse(lse[b:b + 1, h:h + 1, rows], rl, what=f"{name} lse")


# ---------------------------------------------------------------- score variants
@pytest.mark.parametrize("B,H,N,D,window,alibi,dtype", [
    (1, 2, 1000, 64, 256, False, "f16"),
    (1, 2, 700, 128, 256, False, "bf16"),
    (2, 3, 513, 64, 100, False, "bf16"),    # window below one tile
    (1, 2, 600, 64, 1, False, "f16"),       # own key only
    (1, 4, 900, 64, 0, True, "f16"),
    (1, 2, 640, 128, 0, True, "bf16"),
    (1, 3, 1100, 64, 300, True, "f16"),     # window and ALiBi together
    (1, 2, 256, 128, 5000, False, "bf16"),  # window wider than the sequence = causal
    (1, 2, 2600, 64, 1500, False, "f16"),   # a wide window at D = 64: one CTA per unit
    (1, 2, 1300, 64, 1024, True, "bf16"),   # the widest window the persistent kernel takes
])
def test_variants(rf, B, H, N, D, window, alibi, dtype):
    q, k, v = inputs.attn_inputs(B, H, H, N, N, D, dtype, seed=N + window)
    scale = float(np.float32(1 / np.sqrt(D)))
    slopes = oracle.alibi_slopes(H) if alibi else None
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, window=window,
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda() if alibi else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, scale, True, window=window, alibi_slopes=slopes)
    check16(o.cpu(), ro, f"variant W={window} alibi={alibi}")
    check_lse(lse.cpu(), rl, what="variant lse")


@pytest.mark.parametrize("dtype,scale,N,window", [
    ("f16", 0.125, 700, 0),
    ("bf16", 0.125, 700, 0),
    ("f16", 1e-3, 700, 0),     # the bias dominates the scores
    ("f16", 1e-9, 700, 0),     # scores vanish: the bias alone decides
    ("bf16", 1e-9, 700, 0),
    ("f16", 0.125, 2600, 1500),  # a wide window (one CTA per unit) with ALiBi
])
def test_alibi_across_scales(rf, dtype, scale, N, window):
    """ALiBi at D = 64 from the usual score scale down to one where the linear
    bias is all that is left, and with a window too wide for the persistent kernel."""
    H = 3
    q, k, v = inputs.attn_inputs(1, H, H, N, N, 64, dtype, seed=N + H)
    slopes = oracle.alibi_slopes(H)
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, window=window,
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, float(np.float32(scale)), True, window=window, alibi_slopes=slopes)
    check16(o.cpu(), ro, f"ALiBi {dtype} scale={scale}")
    check_lse(lse.cpu(), rl, what="ALiBi lse")


@pytest.mark.parametrize("window,alibi", [(7, False), (0, True), (40, True)])
def test_variants_f32_path(rf, window, alibi):
    q, k, v = inputs.attn_inputs(1, 2, 2, 150, 150, 64, "f32", seed=5)
    slopes = oracle.alibi_slopes(2) if alibi else None
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=0.125, causal=True, window=window,
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda() if alibi else None)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, 0.125, True, window=window, alibi_slopes=slopes)
    from _parity import check32
    check32(o.cpu(), ro, "f32 variant")
    check_lse(lse.cpu(), rl, tol=1e-5 * max(1, np.abs(rl).max()))


def test_package_alibi_slopes_match_oracle(rf):
    np.testing.assert_allclose(rf.alibi_slopes(12, device="cpu").numpy(), oracle.alibi_slopes(12), rtol=1e-7)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["attn_sw256_f16_d64", "attn_causal_alibi_f16_d64"])
def test_variant_workloads_sampled(rf, name):
    w = inputs.WORKLOADS[name]
    d = w.dims
    q, k, v = inputs.make(w)
    scale = float(np.float32(1 / np.sqrt(d["D"])))
    slopes = oracle.alibi_slopes(d["Hq"]) if d.get("alibi") else None
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, window=d.get("window", 0),
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda() if slopes is not None else None)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 255, 256, d["N"] - 1], np.random.default_rng(4).integers(0, d["N"], 60)]))
    for b, h in [(0, 0), (d["B"] - 1, d["Hq"] - 1)]:
        ro, rl = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], scale, True,
                                  rows=rows, window=d.get("window", 0),
                                  alibi_slopes=slopes[h:h + 1] if slopes is not None else None)
        check16(o[b:b + 1, h:h + 1, rows].cpu(), ro, name)
        check_lse(lse[b:b + 1, h:h + 1, rows].cpu(), rl, what=name)


# ---------------------------------------------------------------- split tail
def expected_tail_plan(B, Hq, Nq, Nk, sms):
    """Units of 256 query rows; the last units mod sms are split into min(sms // tail, key tiles) pieces."""
    units = -(-Nq // 256) * B * Hq
    tail = units % sms
    n_split = min(sms // tail, -(-Nk // 128)) if tail else 1
    return (tail, n_split) if tail and n_split >= 2 else (0, 1)


def run_ex(rf, q, k, v, scale, workspace):
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    rf.rf_attn_fwd_ex(q, k, v, o, lse, scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,D,dtype", [
    (1, 8, 8, 1024, 1024, 64, "f16"),    # 32 units: all in the tail
    (1, 1, 1, 256, 4096, 64, "bf16"),    # one unit split into one key tile per piece
    (1, 3, 1, 300, 1000, 128, "bf16"),   # GQA, ragged query rows and keys
    (2, 4, 2, 512, 640, 128, "f16"),
])
def test_split_tail_matches_oracle_and_unsplit(rf, B, Hq, Hkv, Nq, Nk, D, dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tail, n_split = expected_tail_plan(B, Hq, Nq, Nk, sms)
    assert tail > 0, "the case must exercise the split"
    nbytes = rf.rf_attn_fwd_workspace_bytes(B, Hq, Nq, Nk, D, False, inputs.DTYPES[dtype])
    o_bytes = (tail * 256 * n_split * D * 4 + 255) // 256 * 256
    assert nbytes == o_bytes + tail * 256 * n_split * 4
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, Nq, Nk, D, dtype, seed=B * 1000 + Nq + Nk)
    scale = float(np.float32(1 / np.sqrt(D)))
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # stale contents must not matter
    o_split, lse_split = run_ex(rf, q, k, v, scale, ws)
    o_whole, lse_whole = run_ex(rf, q, k, v, scale, None)
    ro, rl = oracle.attention(q, k, v, scale, False)
    check16(o_split, ro, "split tail")
    check_lse(lse_split, rl, what="split tail lse")
    check16(o_whole, ro, "unsplit")
    # the two schedules differ only in rounding order (fp32 partials merged, then one 16-bit rounding)
    assert np.abs(to64(o_split) - to64(o_whole)).max() <= 2e-2
    assert np.abs(to64(lse_split) - to64(lse_whole)).max() <= 1e-3


def test_split_tail_rejects_short_workspace(rf):
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 8, 8, 1024, 1024, 64, "f16", seed=5))
    n = rf.rf_attn_fwd_workspace_bytes(1, 8, 1024, 1024, 64, False, torch.float16)
    assert n > 0
    o = torch.empty_like(q)
    with pytest.raises(rf.RFError, match="workspace"):
        rf.rf_attn_fwd_ex(q, k, v, o, workspace=torch.empty(n - 16, dtype=torch.uint8, device="cuda"))


def test_no_split_cases_need_no_workspace(rf):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rf.rf_attn_fwd_workspace_bytes(1, sms, 256, 1024, 64, False, torch.float16) == 0  # full last wave
    assert rf.rf_attn_fwd_workspace_bytes(1, 1, 256, 128, 64, False, torch.float16) == 0  # one key tile
    assert rf.rf_attn_fwd_workspace_bytes(1, 8, 1024, 1024, 64, True, torch.float16) == 0  # causal
    assert rf.rf_attn_fwd_workspace_bytes(1, 8, 1024, 1024, 64, False, torch.float32) == 0  # fp32 path


@pytest.mark.parametrize("B,Hq,Hkv,N,window,alibi,dtype", [
    (3, 32, 8, 1300, 200, False, "f16"),   # GQA, ragged last unit
    (2, 40, 40, 850, 1, True, "bf16"),     # the last unit's second query tile sees no key tile
    (8, 48, 48, 512, 64, False, "f16"),    # about five units per CTA
])
def test_window_units_walked_by_persistent_ctas(rf, B, Hq, Hkv, N, window, alibi, dtype):
    """D = 64 sliding windows run one CTA per SM over a list of units, so these
    shapes (several units per CTA) cross every item boundary of the schedule:
    Q buffers, K/V ring slots and barrier phases carried from unit to unit."""
    q, k, v = inputs.attn_inputs(B, Hq, Hkv, N, N, 64, dtype, seed=N + window + Hq)
    scale = float(np.float32(1 / np.sqrt(64)))
    slopes = oracle.alibi_slopes(Hq) if alibi else None
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, window=window,
                          alibi_slopes=torch.tensor(slopes, dtype=torch.float32).cuda() if alibi else None)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, N - 1], np.random.default_rng(N).integers(0, N, 40)]))
    G = Hq // Hkv
    for b, h in [(0, 0), (B // 2, Hq // 2 + 1), (B - 1, Hq - 1)]:
        ro, rl = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h // G:h // G + 1], v[b:b + 1, h // G:h // G + 1],
                                  scale, True, rows=rows, window=window,
                                  alibi_slopes=slopes[h:h + 1] if alibi else None)
        check16(o[b:b + 1, h:h + 1, rows].cpu(), ro, f"persistent window b={b} h={h}")
        check_lse(lse[b:b + 1, h:h + 1, rows].cpu(), rl, what="persistent window lse")
    assert np.isfinite(to64(o.cpu())).all()


@pytest.mark.slow
def test_window_grid_widens_past_the_unit_list(rf):
    """A CTA's unit list holds 1024 units, so with more than 1024 units per SM the
    windowed kernel launches more CTAs than SMs: here 163,840 units of 256 rows
    (5.4 GB per tensor)."""
    B, H, N, window = 64, 64, 10240, 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H * (N // 256) > 1024 * sms
    g = torch.Generator(device="cuda").manual_seed(11)
    q, k, v = (torch.randn(B, H, N, 64, device="cuda", generator=g, dtype=torch.float16) for _ in range(3))
    o, lse = rf.attention(q, k, v, scale=0.125, causal=True, window=window)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 255, 256, N - 1], np.random.default_rng(5).integers(0, N, 24)]))
    for b, h in [(0, 0), (B // 2, 17), (B - 1, H - 1)]:
        ro, rl = oracle.attention(q[b:b + 1, h:h + 1].cpu(), k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu(),
                                  0.125, True, rows=rows, window=window)
        check16(o[b:b + 1, h:h + 1, rows].cpu(), ro, f"widened grid b={b} h={h}")
        check_lse(lse[b:b + 1, h:h + 1, rows].cpu(), rl, what="widened grid lse")
    del q, k, v, o, lse


@pytest.mark.parametrize("N,window", [(600, 1), (640, 1), (300, 1), (600, 100), (513, 2)])
def test_window_with_query_tile_past_the_end(rf, N, window):
    """The last unit's second query tile lies wholly past N and a narrow window
    leaves it no key tile: it must finish without waiting for a PV that never
    comes (the post-test check fails on any recorded wait timeout)."""
    q, k, v = inputs.attn_inputs(1, 2, 1, N, N, 64, "f16", seed=N + window)
    scale = float(np.float32(1 / np.sqrt(64)))
    o, lse = rf.attention(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=True, window=window)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, scale, True, window=window)
    check16(o.cpu(), ro, f"window={window} N={N}")
    check_lse(lse.cpu(), rl, what="lse")
    assert rf.rf_device_status(clear=False) == rf.RF_OK
