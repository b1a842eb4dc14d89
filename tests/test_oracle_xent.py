"""Pins for the softmax cross-entropy oracle (CPU only).

Definition: a cascade like attention's safe softmax -- row max, sum of
exponentials, then the loss lse - z_target ("Operator Fusion" guide, section 3:
softmax + cross-entropy is fusible)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_brute_force():
    z = _rand((4, 9), 1) * 3
    t = np.array([0, 8, 3, 5])
    loss, lse, grad = oracle.softmax_xent(z, t)
    for i in range(4):
        ssum = math.fsum(math.exp(v) for v in z[i])
        assert abs(math.log(ssum) - lse[i]) < 1e-12
        assert abs(math.log(ssum) - z[i, t[i]] - loss[i]) < 1e-12
        for j in range(9):
            ref = math.exp(z[i, j]) / ssum - (1.0 if j == t[i] else 0.0)
            assert abs(ref - grad[i, j]) < 1e-12


def test_uniform_logits_give_log_v():
    z = np.full((3, 1000), 2.5)
    loss, lse, grad = oracle.softmax_xent(z, np.array([0, 500, 999]))
    np.testing.assert_allclose(loss, math.log(1000), atol=1e-12)
    np.testing.assert_allclose(lse, 2.5 + math.log(1000), atol=1e-12)
    np.testing.assert_allclose(grad.sum(-1), 0.0, atol=1e-12)


def test_dominant_target_gives_zero_loss_and_shift_invariance():
    z = _rand((2, 50), 2)
    z[0, 7] = 200.0
    z[1, 3] = 150.0
    loss, _, _ = oracle.softmax_xent(z, np.array([7, 3]))
    np.testing.assert_allclose(loss, 0.0, atol=1e-12)
    z2 = _rand((2, 50), 3)
    l1, s1, g1 = oracle.softmax_xent(z2, np.array([1, 2]))
    l2, s2, g2 = oracle.softmax_xent(z2 + 40.0, np.array([1, 2]))
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    np.testing.assert_allclose(s2 - s1, 40.0, atol=1e-12)
    np.testing.assert_allclose(g1, g2, atol=1e-12)


def test_ignore_index_and_gradient_rows():
    z = _rand((3, 20), 4)
    loss, _, grad = oracle.softmax_xent(z, np.array([5, -100, 19]))
    assert loss[1] == 0.0 and (grad[1] == 0).all()
    np.testing.assert_allclose(grad[[0, 2]].sum(-1), 0.0, atol=1e-12)
    assert grad[0, 5] < 0 and (np.delete(grad[0], 5) > 0).all()


def test_torch_second_opinion():
    z = torch.randn(6, 333, dtype=torch.float64, generator=torch.Generator().manual_seed(0)) * 4
    t = torch.randint(0, 333, (6,), generator=torch.Generator().manual_seed(1))
    t[2] = -100
    ref = torch.nn.functional.cross_entropy(z, t, reduction="none", ignore_index=-100)
    zz = z.clone().requires_grad_(True)
    torch.nn.functional.cross_entropy(zz, t, reduction="sum", ignore_index=-100).backward()
    loss, lse, grad = oracle.softmax_xent(z.numpy(), t.numpy())
    np.testing.assert_allclose(loss, ref.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(z, -1).numpy(), atol=1e-12)
    np.testing.assert_allclose(grad, zz.grad.numpy(), atol=1e-12)


def test_incremental_form_reaches_plain_result():
    """Online max/sum over blocks of the row (RedFuser, Figure 4) in fp64 equals
    the plain two-pass log-sum-exp."""
    z = _rand((1, 1001), 5) * 6
    _, lse, _ = oracle.softmax_xent(z, np.array([0]))
    m, l = -np.inf, 0.0
    for j0 in range(0, 1001, 64):
        blk = z[0, j0:j0 + 64]
        mn = max(m, blk.max())
        l = l * math.exp(m - mn) + np.exp(blk - mn).sum() if np.isfinite(m) else np.exp(blk - mn).sum()
        m = mn
    assert abs(m + math.log(l) - lse[0]) < 1e-12
