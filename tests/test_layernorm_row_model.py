"""CPU model of one row of the fused residual + LayerNorm kernel (ln_fused.cu).

The kernel forms both statistics levels in one pass as running sums about a
shift K (the mean of the row's first 16-byte vector): S1 = sum(h - K) and
S2 = sum((h - K)^2), in fp32, per thread over its 16-byte vectors, then summed
across the lanes of a warp (xor butterfly) and across the row's warps.  With
d = S1/n and var = S2/n - d^2, a row whose shift lies more than one standard
deviation from its mean (d^2 > var) recomputes M2 = sum((h - K - d)^2) from the
values it holds.  The output is y = ((h - K) - d) * (gamma * rsqrt(var + eps)) + beta.

This module restates that arithmetic in numpy float32, in the kernel's order,
and checks it against the fp64 oracle within the fp32 bound (1e-5 relative) on
rows built to defeat a one-pass variance: a large common mean, an outlier among
the first elements, a shift just inside and just outside the threshold.  A
planted mistake (no re-centring) must fail.  The GPU tests check the kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import check32

f32 = np.float32


def _thread_sums(vals, tpr, vpt, pairs):
    """Per-thread sums of `vals` [n] in the kernel's layout and order: thread t
    holds 16-byte vectors t, t + tpr, ...; each packed lane sums its elements
    in sequence; the two lanes are then added.  Returns [tpr] float32."""
    per_vec = 2 * pairs
    nvec = vals.size // per_vec
    v = vals.reshape(nvec, pairs, 2)
    out = np.zeros(tpr, dtype=f32)
    for t in range(tpr):
        acc = np.zeros(2, dtype=f32)
        for i in range(vpt):
            c = t + i * tpr
            if c >= nvec:
                continue
            for k in range(pairs):
                acc = (acc + v[c, k]).astype(f32)
        out[t] = f32(acc[0] + acc[1])
    return out


def _row_merge(per_thread):
    """Xor-butterfly within each warp, then the warps in order."""
    w = per_thread.reshape(-1, 32).copy()
    for o in (16, 8, 4, 2, 1):
        w = (w + w[:, np.arange(32) ^ o]).astype(f32)
    tot = f32(0.0)
    for j in range(w.shape[0]):
        tot = f32(tot + w[j, 0]) if j else w[j, 0]
    return tot


def model_row(h, gamma, beta, eps, pairs=2, recentre=True):
    """One fp32 row (h = x + r already formed), fp32 layout (2 pairs per vector)."""
    h = h.astype(f32)
    n = h.size
    nvec = n // (2 * pairs)
    vpt = 4 if nvec >= 128 else (2 if nvec >= 64 else 1)
    tpr = -(-nvec // vpt)
    tpr = (tpr + 31) & ~31
    first = h[:2 * pairs].reshape(pairs, 2)
    w = pairs
    while w > 1:
        w //= 2
        first = (first[:w] + first[w:2 * w]).astype(f32)
    K = f32(f32(first[0, 0] + first[0, 1]) * f32(1.0 / (2 * pairs)))
    d = (h - K).astype(f32)
    a1 = _row_merge(_thread_sums(d, tpr, vpt, pairs))
    a2 = _row_merge(_thread_sums((d * d).astype(f32), tpr, vpt, pairs))
    inv = f32(1.0 / n)
    mk = f32(a1 * inv)
    var = max(f32(f32(a2 * inv) - f32(mk * mk)), f32(0.0))
    took = False
    if recentre and mk * mk > var:
        e = (d - mk).astype(f32)
        var = f32(_row_merge(_thread_sums((e * e).astype(f32), tpr, vpt, pairs)) * inv)
        took = True
    rstd = f32(1.0 / np.sqrt(np.float64(var) + eps))
    a = (gamma.astype(f32) * rstd).astype(f32)
    y = ((d - mk).astype(f32) * a + beta.astype(f32)).astype(f32)
    return y, took


def _rows(kind, n=4096, seed=0):
    g = np.random.default_rng(seed)
    h = g.standard_normal(n)
    if kind == "large_mean":            # mean 1000, sigma 0.01
        h = 1000.0 + 0.01 * h
    elif kind == "outlier_first":       # first element far outside the row
        h = 0.01 * h
        h[0] = 1000.0
    elif kind == "shift_inside":        # first vector 0.9 sigma off the row mean
        h[:4] = 0.9
    elif kind == "shift_outside":       # 1.1 sigma off: the re-centring path
        h[:4] = 1.1
    elif kind == "big_offset_first_vector":
        h[:4] = 40.0
    return h.astype(f32)


CASES = [("plain", False), ("large_mean", False), ("outlier_first", True), ("shift_inside", False),
         ("shift_outside", True), ("big_offset_first_vector", True)]


@pytest.mark.parametrize("kind,expect_recentre", CASES)
def test_model_row_meets_fp32_bound(kind, expect_recentre):
    n = 4096
    h = _rows(kind, n)
    g = np.random.default_rng(1).uniform(0.5, 1.5, n).astype(f32)
    b = (0.1 * np.random.default_rng(2).standard_normal(n)).astype(f32)
    y, took = model_row(h, g, b, 1e-5)
    assert took == expect_recentre, kind
    t = lambda a: torch.from_numpy(a[None, :])
    ref, _ = oracle.layernorm(t(h), torch.zeros(1, n), t(g), t(b), 1e-5)
    check32(y[None, :], ref, kind)


def test_constant_row_gives_beta_exactly():
    n = 1024
    h = np.full(n, 1.0 + 2.0 ** -20, dtype=f32)
    b = (0.1 * np.random.default_rng(3).standard_normal(n)).astype(f32)
    y, took = model_row(h, np.ones(n, dtype=f32), b, 1e-5)
    assert not took
    np.testing.assert_array_equal(y, b)


def test_planted_mistake_without_recentring_fails():
    # An outlier among the first elements makes the one-pass M2 cancel: without
    # the second reduction the fp32 bound fails.
    n = 4096
    h = _rows("big_offset_first_vector", n)
    h[:4] = 3000.0
    g = np.ones(n, dtype=f32)
    b = np.zeros(n, dtype=f32)
    t = lambda a: torch.from_numpy(a[None, :])
    ref, _ = oracle.layernorm(t(h), torch.zeros(1, n), t(g), t(b), 1e-5)
    y_ok, _ = model_row(h, g, b, 1e-5)
    check32(y_ok[None, :], ref, "with re-centring")
    y_bad, _ = model_row(h, g, b, 1e-5, recentre=False)
    with pytest.raises(AssertionError):
        check32(y_bad[None, :], ref, "planted: no re-centring")
