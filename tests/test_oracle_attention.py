"""Pins for the attention / decode oracle (CPU only).

Each test checks the oracle against something other than itself: brute force
in pure Python, closed forms, invariants fixed by the definition (RedFuser,
Abstract: safe softmax followed by GEMM; "Operator Fusion" guide, section 2,
Pattern 4), and a library second opinion.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def brute_attention(q, k, v, scale, causal):
    """Pure-Python loops, math.fsum / math.exp, straight from the definition."""
    B, Hq, Nq, D = q.shape
    Hkv, Nk, Dv = k.shape[1], k.shape[2], v.shape[3]
    g = Hq // Hkv
    o = np.zeros((B, Hq, Nq, Dv))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            for i in range(Nq):
                keys = [j for j in range(Nk) if (not causal or j <= i)]
                s = [scale * math.fsum(q[b, h, i, d] * k[b, kh, j, d] for d in range(D)) for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = math.fsum(e)
                for d in range(Dv):
                    o[b, h, i, d] = math.fsum(e[t] * v[b, kh, keys[t], d] for t in range(len(keys))) / tot
                lse[b, h, i] = m + math.log(tot)
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal", [
    (1, 1, 1, 5, 3, False),
    (1, 1, 1, 7, 4, True),
    (2, 4, 2, 6, 8, False),   # GQA 4q/2kv
    (1, 4, 2, 9, 5, True),    # GQA + causal
    (1, 3, 3, 16, 8, False),
])
def test_brute_force(B, Hq, Hkv, N, D, causal):
    q = _rand((B, Hq, N, D), 1)
    k = _rand((B, Hkv, N, D), 2)
    v = _rand((B, Hkv, N, D), 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attention(q, k, v, scale, causal)
    ob, lb = brute_attention(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_mpmath_50_digits():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    q = _rand((1, 1, 3, 4), 7) * 3
    k = _rand((1, 1, 4, 4), 8) * 3
    v = _rand((1, 1, 4, 2), 9)
    o, lse = oracle.attention(q, k, v, 0.5, False)
    for i in range(3):
        s = [mp.mpf(0.5) * mp.fsum(mp.mpf(q[0, 0, i, d]) * mp.mpf(k[0, 0, j, d]) for d in range(4)) for j in range(4)]
        z = mp.fsum(mp.e ** x for x in s)
        assert abs(float(mp.log(z)) - lse[0, 0, i]) < 1e-13
        for d in range(2):
            ref = mp.fsum(mp.e ** s[j] * mp.mpf(v[0, 0, j, d]) for j in range(4)) / z
            assert abs(float(ref) - o[0, 0, i, d]) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    # With V = identity (Dv = Nk) the output row IS the softmax row.
    N = 12
    q = _rand((1, 2, N, 6), 4) * 2
    k = _rand((1, 2, N, 6), 5) * 2
    v = np.broadcast_to(np.eye(N), (1, 2, N, N)).copy()
    o, _ = oracle.attention(q, k, v, 0.4, causal)
    np.testing.assert_allclose(o.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
    assert (o >= 0).all()
    if causal:
        # masked weights are exactly zero
        assert np.all(np.triu(o[0, 0], k=1) == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_rows(causal):
    q = _rand((2, 4, 10, 8), 6)
    k = _rand((2, 2, 10, 8), 7)
    row = _rand((8,), 8)
    v = np.broadcast_to(row, (2, 2, 10, 8)).copy()
    o, _ = oracle.attention(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), rtol=0, atol=1e-12)


def test_one_hot_dominant_score():
    rng = np.random.default_rng(11)
    N, D = 8, 16
    k = rng.standard_normal((1, 1, N, D))
    v = rng.standard_normal((1, 1, N, D))
    targets = rng.permutation(N)
    # q_i = c * k_{t(i)} makes score (i, t(i)) exceed every other by >> 40
    q = np.stack([50.0 * k[0, 0, t] for t in targets])[None, None]
    o, _ = oracle.attention(q, k, v, 1.0, False)
    s = q[0, 0] @ k[0, 0].T
    for i, t in enumerate(targets):
        others = np.delete(s[i], t)
        assert s[i, t] - others.max() > 40
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, t], rtol=0, atol=1e-12)


def test_zero_query_closed_form():
    N, D = 11, 5
    v = _rand((1, 1, N, D), 12)
    k = _rand((1, 1, N, D), 13)
    q = np.zeros((1, 1, N, D))
    o, lse = oracle.attention(q, k, v, 0.7, False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (N, D)), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-12)
    o, lse = oracle.attention(q, k, v, 0.7, True)
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], prefix, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-12)


def test_causal_row_zero():
    q = _rand((1, 2, 6, 4), 14)
    k = _rand((1, 2, 6, 4), 15)
    v = _rand((1, 2, 6, 4), 16)
    o, lse = oracle.attention(q, k, v, 0.9, True)
    for h in range(2):
        np.testing.assert_allclose(o[0, h, 0], v[0, h, 0], atol=1e-12)
        np.testing.assert_allclose(lse[0, h, 0], 0.9 * q[0, h, 0] @ k[0, h, 0], atol=1e-12)


def test_key_permutation_invariance():
    q = _rand((1, 2, 7, 4), 17)
    k = _rand((1, 2, 9, 4), 18)
    v = _rand((1, 2, 9, 3), 19)
    perm = np.random.default_rng(20).permutation(9)
    o1, l1 = oracle.attention(q, k, v, 0.5, False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_score_shift_invariance(causal):
    # Append a feature a to every query and 1 to every key: each score of a row
    # grows by scale*a.  O must not move; LSE must move by exactly scale*a.
    N, D, scale = 8, 4, 0.5
    q = _rand((1, 1, N, D), 21)
    k = _rand((1, 1, N, D), 22)
    v = _rand((1, 1, N, D), 23)
    a = _rand((N,), 24) * 10
    q2 = np.concatenate([q, a[None, None, :, None]], axis=-1)
    k2 = np.concatenate([k, np.ones((1, 1, N, 1))], axis=-1)
    o1, l1 = oracle.attention(q, k, v, scale, causal)
    o2, l2 = oracle.attention(q2, k2, v, scale, causal)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * a[None, None, :], atol=1e-12)


def test_gqa_head_map_consecutive_groups():
    # Hq = 4, Hkv = 2: heads 0,1 read kv head 0; heads 2,3 read kv head 1.
    q = _rand((1, 4, 5, 3), 25)
    k = _rand((1, 2, 5, 3), 26)
    v = _rand((1, 2, 5, 3), 27)
    o, _ = oracle.attention(q, k, v, 1.0, False)
    for h in range(4):
        oh, _ = oracle.attention(q[:, h:h + 1], k[:, h // 2:h // 2 + 1], v[:, h // 2:h // 2 + 1], 1.0, False)
        np.testing.assert_allclose(o[:, h:h + 1], oh, atol=0)


def test_rows_subset_matches_full():
    q = _rand((1, 2, 20, 4), 28)
    k = _rand((1, 1, 20, 4), 29)
    v = _rand((1, 1, 20, 4), 30)
    rows = [0, 3, 19, 7]
    for causal in (False, True):
        of, lf = oracle.attention(q, k, v, 0.5, causal)
        os_, ls = oracle.attention(q, k, v, 0.5, causal, rows=rows)
        np.testing.assert_allclose(os_, of[:, :, rows], atol=0)
        np.testing.assert_allclose(ls, lf[:, :, rows], atol=0)


def test_empty_keys():
    q = _rand((1, 1, 3, 4), 31)
    k = np.zeros((1, 1, 0, 4))
    o, lse = oracle.attention(q, k, k, 1.0, False)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_torch_sdpa_second_opinion():
    q = torch.randn(2, 4, 33, 16, dtype=torch.float64, generator=torch.Generator().manual_seed(0))
    k = torch.randn(2, 2, 33, 16, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
    v = torch.randn(2, 2, 33, 16, dtype=torch.float64, generator=torch.Generator().manual_seed(2))
    for causal in (False, True):
        kk = k.repeat_interleave(2, dim=1)
        vv = v.repeat_interleave(2, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=causal, scale=0.25)
        o, _ = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.25, causal)
        np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
        s = (q @ kk.transpose(-1, -2)) * 0.25
        if causal:
            s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
        _, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.25, causal)
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_incremental_form_reaches_plain_result(causal):
    """The fused single-loop incremental form (RedFuser, Figures 3-4) -- a running
    max m, running sum l and running O rescaled by exp(m_old - m_new) as each
    key block arrives -- written here in fp64 reaches the oracle's plain result."""
    N, D, blk = 37, 8, 5
    q = _rand((1, 1, N, D), 32)
    k = _rand((1, 1, N, D), 33)
    v = _rand((1, 1, N, D), 34)
    scale = 0.35
    ref_o, ref_l = oracle.attention(q, k, v, scale, causal)
    for i in range(N):
        m, l, acc = -np.inf, 0.0, np.zeros(D)
        for j0 in range(0, N, blk):
            js = [j for j in range(j0, min(N, j0 + blk)) if not causal or j <= i]
            if not js:
                continue
            s = scale * (k[0, 0, js] @ q[0, 0, i])
            m_new = max(m, s.max())
            alpha = math.exp(m - m_new) if np.isfinite(m) else 0.0
            p = np.exp(s - m_new)
            l = alpha * l + p.sum()
            acc = alpha * acc + p @ v[0, 0, js]
            m = m_new
        np.testing.assert_allclose(acc / l, ref_o[0, 0, i], atol=1e-12)
        assert abs(m + math.log(l) - ref_l[0, 0, i]) < 1e-12


def test_decode_matches_attention_with_one_query():
    q = _rand((2, 8, 1, 16), 35)
    k = _rand((2, 2, 40, 16), 36)
    v = _rand((2, 2, 40, 16), 37)
    o, lse = oracle.decode(q, k, v, 0.25)
    o2, l2 = oracle.attention(q, k, v, 0.25, False)
    np.testing.assert_allclose(o, o2[:, :, 0], atol=0)
    np.testing.assert_allclose(lse, l2[:, :, 0], atol=0)
    o3, l3 = oracle.decode(q[:, :, 0], k, v, 0.25)
    np.testing.assert_allclose(o3, o, atol=0)


# ---------------------------------------------------------------- score variants
def brute_variant(q, k, v, scale, window, slopes):
    B, Hq, N, D = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, N))
    for h in range(Hq):
        for i in range(N):
            keys = [j for j in range(N) if j <= i and (not window or j > i - window)]
            s = [scale * math.fsum(q[0, h, i, d] * k[0, h, j, d] for d in range(D))
                 + (slopes[h] * (j - i) if slopes is not None else 0.0) for j in keys]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            t = math.fsum(e)
            for d in range(D):
                o[0, h, i, d] = math.fsum(e[a] * v[0, h, keys[a], d] for a in range(len(keys))) / t
            lse[0, h, i] = m + math.log(t)
    return o, lse


@pytest.mark.parametrize("window,alibi", [(3, False), (1, False), (0, True), (4, True)])
def test_variants_brute_force(window, alibi):
    q, k, v = _rand((1, 2, 9, 4), 40), _rand((1, 2, 9, 4), 41), _rand((1, 2, 9, 4), 42)
    slopes = oracle.alibi_slopes(2) if alibi else None
    o, lse = oracle.attention(q, k, v, 0.5, True, window=window, alibi_slopes=slopes)
    ob, lb = brute_variant(q, k, v, 0.5, window, slopes)
    np.testing.assert_allclose(o, ob, atol=1e-12)
    np.testing.assert_allclose(lse, lb, atol=1e-12)


def test_window_limits():
    q, k, v = _rand((1, 1, 20, 4), 43), _rand((1, 1, 20, 4), 44), _rand((1, 1, 20, 4), 45)
    full, lf = oracle.attention(q, k, v, 0.5, True)
    wide, lw = oracle.attention(q, k, v, 0.5, True, window=20)
    np.testing.assert_allclose(wide, full, atol=0)
    np.testing.assert_allclose(lw, lf, atol=0)
    one, l1 = oracle.attention(q, k, v, 0.5, True, window=1)  # each query sees only its own key
    np.testing.assert_allclose(one[0, 0], v[0, 0], atol=1e-12)
    np.testing.assert_allclose(l1[0, 0], 0.5 * (q[0, 0] * k[0, 0]).sum(-1), atol=1e-12)


def test_alibi_limits_and_slopes():
    q, k, v = _rand((1, 2, 12, 4), 46), _rand((1, 2, 12, 4), 47), _rand((1, 2, 12, 4), 48)
    base, lb = oracle.attention(q, k, v, 0.5, True)
    zero, lz = oracle.attention(q, k, v, 0.5, True, alibi_slopes=np.zeros(2))
    np.testing.assert_allclose(zero, base, atol=0)
    steep, _ = oracle.attention(q, k, v, 0.5, True, alibi_slopes=np.full(2, 500.0))  # bias wins: own key only
    np.testing.assert_allclose(steep[0, :], v[0, :], atol=1e-12)
    s = oracle.alibi_slopes(8)
    np.testing.assert_allclose(s, 2.0 ** (-np.arange(1, 9)), atol=0)
