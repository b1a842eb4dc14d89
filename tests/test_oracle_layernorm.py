"""Pins for the residual + LayerNorm oracle (CPU only).

Definition: "Operator Fusion" guide, section 2, Pattern 2 (mean -> variance ->
normalise) and section 4 (residual added first, eps inside the square root,
biased variance, affine gamma/beta).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def brute_ln(x, r, g, b, eps):
    y = np.zeros_like(x)
    for i in range(x.shape[0]):
        h = [x[i, j] + r[i, j] for j in range(x.shape[1])]
        n = len(h)
        mu = math.fsum(h) / n
        var = math.fsum((t - mu) ** 2 for t in h) / n
        for j in range(n):
            y[i, j] = (h[j] - mu) / math.sqrt(var + eps) * g[j] + b[j]
    return y


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 7), (4, 16), (2, 33)])
def test_brute_force(rows, cols):
    x, r = _rand((rows, cols), 1), _rand((rows, cols), 2)
    g, b = _rand((cols,), 3), _rand((cols,), 4)
    y, h = oracle.layernorm(x, r, g, b, 1e-5)
    np.testing.assert_allclose(y, brute_ln(x, r, g, b, 1e-5), atol=1e-12)
    np.testing.assert_array_equal(h, x + r)


def test_pre_affine_mean_zero_biased_variance():
    x, r = _rand((8, 64), 5) * 3 + 1, _rand((8, 64), 6)
    eps = 1e-5
    y, h = oracle.layernorm(x, r, np.ones(64), np.zeros(64), eps)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-12)
    var = h.var(-1)  # numpy default ddof=0: biased
    np.testing.assert_allclose((y ** 2).mean(-1), var / (var + eps), atol=1e-12)


def test_constant_row_gives_beta():
    x = np.full((2, 10), 3.25)
    r = np.full((2, 10), -1.0)
    g, b = _rand((10,), 7), _rand((10,), 8)
    y, _ = oracle.layernorm(x, r, g, b, 1e-5)
    np.testing.assert_allclose(y, np.broadcast_to(b, y.shape), atol=1e-12)


def test_plus_minus_a_row():
    a, eps = 0.7, 1e-3
    x = np.array([[a, -a, a, -a, -a, a]])
    g, b = _rand((6,), 9), _rand((6,), 10)
    y, _ = oracle.layernorm(x, np.zeros_like(x), g, b, eps)
    np.testing.assert_allclose(y[0], np.sign(x[0]) * a / math.sqrt(a * a + eps) * g + b, atol=1e-12)


def test_shift_invariance():
    x, r = _rand((3, 20), 11), _rand((3, 20), 12)
    g, b = _rand((20,), 13), _rand((20,), 14)
    y1, _ = oracle.layernorm(x, r, g, b, 1e-5)
    y2, _ = oracle.layernorm(x + 5.0, r, g, b, 1e-5)
    np.testing.assert_allclose(y1, y2, atol=1e-11)


def test_residual_is_added_not_swapped():
    # The residual and x enter symmetrically through h = x + r; swapping them must
    # not change y, while dropping r must.
    x, r = _rand((2, 12), 15), _rand((2, 12), 16)
    g, b = np.ones(12), np.zeros(12)
    y1, _ = oracle.layernorm(x, r, g, b, 1e-5)
    y2, _ = oracle.layernorm(r, x, g, b, 1e-5)
    y3, _ = oracle.layernorm(x, 0 * r, g, b, 1e-5)
    np.testing.assert_allclose(y1, y2, atol=1e-12)
    assert np.abs(y1 - y3).max() > 0.1


def test_torch_layer_norm_second_opinion():
    x = torch.randn(5, 48, dtype=torch.float64, generator=torch.Generator().manual_seed(0))
    r = torch.randn(5, 48, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
    g = torch.rand(48, dtype=torch.float64, generator=torch.Generator().manual_seed(2)) + 0.5
    b = torch.randn(48, dtype=torch.float64, generator=torch.Generator().manual_seed(3)) * 0.1
    ref = torch.nn.functional.layer_norm(x + r, (48,), g, b, eps=1e-5)
    y, _ = oracle.layernorm(x.numpy(), r.numpy(), g.numpy(), b.numpy(), 1e-5)
    np.testing.assert_allclose(y, ref.numpy(), atol=1e-12)


def test_welford_chan_incremental_form_reaches_plain_result():
    """The incremental form (RedFuser, Figure 4) of mean -> M2: Welford's update
    per element and Chan et al.'s pairwise combine of partial (n, mean, M2),
    written here in fp64, reaches the oracle's plain two-pass statistics."""
    x = _rand((1, 101), 17) * 4 + 10
    r = np.zeros_like(x)
    y, h = oracle.layernorm(x, r, np.ones(101), np.zeros(101), 1e-5)

    def welford(vals):
        n, mean, m2 = 0, 0.0, 0.0
        for t in vals:
            n += 1
            d = t - mean
            mean += d / n
            m2 += d * (t - mean)
        return n, mean, m2

    def chan(a, b):
        na, ma, qa = a
        nb, mb, qb = b
        n = na + nb
        if n == 0:
            return 0, 0.0, 0.0
        d = mb - ma
        return n, ma + d * nb / n, qa + qb + d * d * na * nb / n

    parts = [welford(h[0, i:i + 13]) for i in range(0, 101, 13)] + [welford([])]
    tot = parts[0]
    for p in parts[1:]:
        tot = chan(tot, p)
    n, mean, m2 = tot
    yy = (h[0] - mean) / math.sqrt(m2 / n + 1e-5)
    np.testing.assert_allclose(yy, y[0], atol=1e-12)


def test_shifted_sums_reach_plain_result():
    """The one-pass form with one shift K for the whole row (its first element):
    S1 = sum(h - K), S2 = sum((h - K)^2) accumulate as plain running sums in any
    partition and order, and mean = K + S1/n, M2 = S2 - S1^2/n is the plain
    two-pass statistics exactly (in fp64, to rounding)."""
    x = _rand((1, 101), 18) * 4 + 10
    y, h = oracle.layernorm(x, np.zeros_like(x), np.ones(101), np.zeros(101), 1e-5)
    row = h[0]
    k = row[0]
    parts = [(float(np.sum(row[i:i + 13] - k)), float(np.sum((row[i:i + 13] - k) ** 2))) for i in range(0, 101, 13)]
    s1 = math.fsum(p[0] for p in parts)
    s2 = math.fsum(p[1] for p in parts)
    n = row.size
    mean, m2 = k + s1 / n, s2 - s1 * s1 / n
    np.testing.assert_allclose(mean, row.mean(), rtol=1e-14)
    np.testing.assert_allclose(m2 / n, np.mean((row - row.mean()) ** 2), rtol=1e-12)
    yy = (row - mean) / math.sqrt(m2 / n + 1e-5)
    np.testing.assert_allclose(yy, y[0], atol=1e-12)


def test_shifted_sums_keep_float32_variance_for_a_large_mean():
    """Why the shift: in float32, the unshifted one-pass formula
    E[h^2] - E[h]^2 cancels catastrophically for a row of mean 1000 and spread
    0.5; sums about the row's first element keep the variance accurate."""
    rng = np.random.default_rng(19)
    row = (1000.0 + 0.5 * rng.standard_normal(4096)).astype(np.float32)
    exact = np.var(row.astype(np.float64))
    n = np.float32(row.size)
    s1 = np.float32(0)
    s2 = np.float32(0)
    k = row[0]
    for v in row:  # float32 running sums, element by element
        d = np.float32(v - k)
        s1 = np.float32(s1 + d)
        s2 = np.float32(s2 + d * d)
    var_shifted = np.float32(s2 / n - (s1 / n) * (s1 / n))
    t1 = np.float32(0)
    t2 = np.float32(0)
    for v in row:
        t1 = np.float32(t1 + v)
        t2 = np.float32(t2 + v * v)
    var_naive = np.float32(t2 / n - (t1 / n) * (t1 / n))
    assert abs(var_shifted - exact) / exact < 1e-3
    assert abs(var_naive - exact) / exact > 1e-2  # the form the shift avoids


# ---------------------------------------------------------------- RMSNorm
def brute_rms(x, r, g, eps):
    y = np.zeros_like(x)
    for i in range(x.shape[0]):
        h = [x[i, j] + r[i, j] for j in range(x.shape[1])]
        ms = math.fsum(t * t for t in h) / len(h)
        for j in range(len(h)):
            y[i, j] = h[j] / math.sqrt(ms + eps) * g[j]
    return y


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 7), (2, 33)])
def test_rms_brute_force(rows, cols):
    x, r, g = _rand((rows, cols), 21), _rand((rows, cols), 22), _rand((cols,), 23)
    y, h = oracle.rmsnorm(x, r, g, 1e-5)
    np.testing.assert_allclose(y, brute_rms(x, r, g, 1e-5), atol=1e-12)
    np.testing.assert_array_equal(h, x + r)


def test_rms_unit_mean_square_and_closed_form():
    x = _rand((6, 40), 24) * 3
    y, _ = oracle.rmsnorm(x, np.zeros_like(x), np.ones(40), 0.0)
    np.testing.assert_allclose((y ** 2).mean(-1), 1.0, atol=1e-12)
    # a constant row c gives c / sqrt(c^2 + eps) * gamma
    c, eps = -1.75, 1e-3
    g = _rand((9,), 25)
    y, _ = oracle.rmsnorm(np.full((1, 9), c), np.zeros((1, 9)), g, eps)
    np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * g, atol=1e-12)


def test_rms_scale_invariance_without_eps():
    x = _rand((3, 16), 26)
    g = _rand((16,), 27)
    y1, _ = oracle.rmsnorm(x, np.zeros_like(x), g, 0.0)
    y2, _ = oracle.rmsnorm(7.5 * x, np.zeros_like(x), g, 0.0)
    np.testing.assert_allclose(y1, y2, atol=1e-12)
    # unlike LayerNorm, a constant shift changes the result
    y3, _ = oracle.rmsnorm(x + 3.0, np.zeros_like(x), g, 0.0)
    assert np.abs(y3 - y1).max() > 0.1


def test_rms_torch_second_opinion():
    x = torch.randn(4, 64, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    r = torch.randn(4, 64, dtype=torch.float64, generator=torch.Generator().manual_seed(6))
    g = torch.rand(64, dtype=torch.float64, generator=torch.Generator().manual_seed(7)) + 0.5
    if not hasattr(torch.nn.functional, "rms_norm"):
        pytest.skip("torch without rms_norm")
    ref = torch.nn.functional.rms_norm(x + r, (64,), g, eps=1e-5)
    y, _ = oracle.rmsnorm(x.numpy(), r.numpy(), g.numpy(), 1e-5)
    np.testing.assert_allclose(y, ref.numpy(), atol=1e-12)
