"""Pins of oracle.rope (rotary position embedding, rotate-half pairing).

Each check holds for rotary embeddings by construction, not by retyping the
oracle: worked values with the angle derived by hand, the same rotation as a
complex multiplication, and the properties that make RoPE a relative position
encoding."""
import numpy as np

import oracle


def test_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((3, 5, 8))
    np.testing.assert_allclose(oracle.rope(x, np.zeros(5)), x, rtol=0, atol=0)


def test_d2_turns_by_the_position_in_radians():
    # D = 2: the only frequency is base^0 = 1, so position p turns (1, 0) by p radians, counter-clockwise
    for p in (1, 2, 7):
        y = oracle.rope(np.array([[1.0, 0.0]]), [p])
        np.testing.assert_allclose(y, [[np.cos(p), np.sin(p)]], rtol=0, atol=1e-15)
    y = oracle.rope(np.array([[0.0, 1.0]]), [1])
    np.testing.assert_allclose(y, [[-np.sin(1.0), np.cos(1.0)]], rtol=0, atol=1e-15)


def test_d4_second_pair_and_its_frequency():
    # D = 4, base 10000: pair 1 is (x_1, x_3) and turns at 10000^(-2/4) = 1/100 rad per position,
    # so at position 100 it has turned by exactly 1 radian while pair 0 (x_0, x_2) turned by 100 radians.
    y = oracle.rope(np.array([[0.0, 1.0, 0.0, 0.0]]), [100], base=10000.0)
    np.testing.assert_allclose(y, [[0.0, np.cos(1.0), 0.0, np.sin(1.0)]], rtol=0, atol=1e-14)
    y = oracle.rope(np.array([[1.0, 0.0, 0.0, 0.0]]), [100], base=10000.0)
    np.testing.assert_allclose(y, [[np.cos(100.0), 0.0, np.sin(100.0), 0.0]], rtol=0, atol=1e-13)


def test_matches_complex_multiplication():
    # pair (a, b) as the complex number a + ib, turned by multiplying with e^{i theta_j}; the angle of pair j
    # at position p is p * base^(-j / (D/2)) (the frequencies form a geometric sequence from 1 down to base^-1+2/D)
    rng = np.random.default_rng(1)
    D, N, base = 16, 9, 500000.0
    x = rng.standard_normal((2, N, D))
    pos = rng.integers(0, 70000, N)
    half = D // 2
    z = x[..., :half] + 1j * x[..., half:]
    ratio = base ** (-1.0 / half)
    theta = pos[:, None] * ratio ** np.arange(half)[None, :]
    w = z * np.exp(1j * theta)
    np.testing.assert_allclose(oracle.rope(x, pos, base=base), np.concatenate([w.real, w.imag], -1),
                               rtol=1e-9, atol=1e-9)


def test_rotation_keeps_pair_norms_and_inverts():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 11, 32))
    pos = rng.integers(0, 9000, 11)
    y = oracle.rope(x, pos)
    np.testing.assert_allclose(y[..., :16] ** 2 + y[..., 16:] ** 2, x[..., :16] ** 2 + x[..., 16:] ** 2, rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(y, -pos), x, rtol=1e-9, atol=1e-9)


def test_scores_depend_only_on_relative_position():
    # <R_m q, R_n k> = <q, R_{n-m} k>: shifting both positions leaves the score unchanged
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((2, 1, 64))
    for m, n, shift in ((3, 10, 1000), (500, 20, 77), (0, 4095, 12345)):
        a = oracle.rope(q, [m]) @ oracle.rope(k, [n]).T
        b = oracle.rope(q, [m + shift]) @ oracle.rope(k, [n + shift]).T
        c = q @ oracle.rope(k, [n - m]).T
        np.testing.assert_allclose(a, b, rtol=1e-9)
        np.testing.assert_allclose(a, c, rtol=1e-9)
