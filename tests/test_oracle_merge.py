"""Pins for the split partition and the log-sum-exp merge oracle (CPU only).

The merge is the incremental combine across splits (RedFuser, Figure 4: a
level's result is updated as each new part arrives; Figure 13, FlashDecoding
IR).  Its plain definition is LSE = ln sum_s exp(lse_s), O = sum_s
exp(lse_s - LSE) O_s; the pins below tie it to the unsplit attention oracle.
"""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("L,S", [(2048, 16), (100, 7), (5, 8), (0, 3), (1, 1), (32768, 16)])
def test_split_bounds_partition(L, S):
    b = oracle.split_bounds(L, S)
    assert len(b) == S and b[0][0] == 0 and b[-1][1] == L
    for (lo, hi), (lo2, _) in zip(b, b[1:]):
        assert hi == lo2 and hi >= lo
    sizes = [hi - lo for lo, hi in b]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("L,S", [(64, 1), (64, 2), (100, 13), (80, 16), (5, 8)])
def test_split_invariance(L, S):
    """Merging the oracle's per-split results equals the unsplit oracle (also when
    some splits are empty: L < S)."""
    q = _rand((2, 4, 1, 8), 1) * 2
    k = _rand((2, 2, L, 8), 2)
    v = _rand((2, 2, L, 8), 3)
    o_ref, lse_ref = oracle.decode(q, k, v, 0.5)
    o_part, lse_part = oracle.decode_partials(q, k, v, 0.5, S)
    o, lse = oracle.lse_merge(o_part, lse_part)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_merge_any_partition():
    # Any partition of the keys (not only contiguous chunks) merges to the whole.
    L = 30
    q = _rand((1, 1, 1, 4), 4)
    k = _rand((1, 1, L, 4), 5)
    v = _rand((1, 1, L, 6), 6)
    groups = [np.arange(0, L, 3), np.arange(1, L, 3), np.arange(2, L, 3), np.array([], dtype=int)]
    o_parts, l_parts = [], []
    for g in groups:
        o_s, l_s = oracle.attention(q, k[:, :, g], v[:, :, g], 1.0, False)
        o_parts.append(o_s[0, 0, 0])
        l_parts.append(l_s[0, 0, 0])
    o, lse = oracle.lse_merge(np.array(o_parts)[None], np.array(l_parts)[None])
    o_ref, l_ref = oracle.decode(q, k, v, 1.0)
    np.testing.assert_allclose(o[0], o_ref[0, 0], atol=1e-12)
    assert abs(lse[0] - l_ref[0, 0]) < 1e-12


def test_merge_brute_force():
    o_part = _rand((3, 5, 4), 7)
    lse_part = _rand((3, 5), 8) * 5
    o, lse = oracle.lse_merge(o_part, lse_part)
    for r in range(3):
        z = math.fsum(math.exp(x) for x in lse_part[r])
        assert abs(math.log(z) - lse[r]) < 1e-12
        for d in range(4):
            ref = math.fsum(math.exp(lse_part[r, s]) * o_part[r, s, d] for s in range(5)) / z
            assert abs(ref - o[r, d]) < 1e-12


def test_merge_large_lse_no_overflow():
    o_part = _rand((2, 4, 3), 9)
    lse_part = np.array([[800.0, 801.0, 799.5, -np.inf], [-1000.0, -999.0, -np.inf, -np.inf]])
    o, lse = oracle.lse_merge(o_part, lse_part)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    w = np.exp(lse_part[0, :3] - 801.0)
    np.testing.assert_allclose(lse[0], 801.0 + math.log(w.sum()), atol=1e-12)
    np.testing.assert_allclose(o[0], (w[:, None] * o_part[0, :3]).sum(0) / w.sum(), atol=1e-12)


def test_merge_single_split_is_identity():
    o_part = _rand((6, 1, 5), 10)
    lse_part = _rand((6, 1), 11)
    o, lse = oracle.lse_merge(o_part, lse_part)
    np.testing.assert_allclose(o, o_part[:, 0], atol=0)
    np.testing.assert_allclose(lse, lse_part[:, 0], atol=1e-15)


def test_merge_all_empty_row():
    o_part = np.zeros((2, 3, 4))
    lse_part = np.full((2, 3), -np.inf)
    lse_part[1, 2] = 0.25
    o_part[1, 2] = 1.5
    o, lse = oracle.lse_merge(o_part, lse_part)
    assert (o[0] == 0).all() and np.isneginf(lse[0])
    np.testing.assert_allclose(o[1], 1.5, atol=0)
    assert lse[1] == 0.25


def test_merge_weights_sum_to_one():
    # With O_s = e_s (one-hot per split) the merged O is the weight vector.
    S = 9
    o_part = np.broadcast_to(np.eye(S), (4, S, S)).copy()
    lse_part = _rand((4, S), 12) * 3
    o, _ = oracle.lse_merge(o_part, lse_part)
    np.testing.assert_allclose(o.sum(-1), 1.0, atol=1e-12)
    np.testing.assert_allclose(o, np.exp(lse_part) / np.exp(lse_part).sum(-1, keepdims=True), atol=1e-12)


def test_table1_operator_algebra():
    """RedFuser, Table 1: each reduce op pairs with a combine op that distributes
    over it -- max with + and + with *.  That distributivity is what lets a running
    result be corrected by one combine step when an earlier level changes."""
    rng = np.random.default_rng(13)
    a, b, c = rng.standard_normal((3, 1000))
    np.testing.assert_array_equal(np.maximum(a, b) + c, np.maximum(a + c, b + c))
    np.testing.assert_array_equal(np.minimum(a, b) + c, np.minimum(a + c, b + c))
    np.testing.assert_allclose((a + b) * c, a * c + b * c, atol=1e-12)
    # exp turns the (max, +) correction into the (+, *) one: exp(x - m') = exp(x - m) * exp(m - m')
    m, m2 = 0.3, 1.7
    np.testing.assert_allclose(np.exp(a - m2), np.exp(a - m) * np.exp(m - m2), rtol=1e-14)
    # Table 1 footnote: a product is a signed power of two of a sum of logs
    x = rng.uniform(-2, 2, 7)
    np.testing.assert_allclose(np.prod(x), np.prod(np.sign(x)) * 2.0 ** np.sum(np.log2(np.abs(x))), rtol=1e-12)
