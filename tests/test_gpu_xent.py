"""GPU parity of rf_softmax_xent (loss, LSE, gradient) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check32, to64

pytestmark = pytest.mark.gpu


def run(rf, logits, targets, want_grad=True):
    res = rf.softmax_xent(logits.cuda(), targets.cuda(), want_grad=want_grad)
    torch.cuda.synchronize()
    return [t.cpu() if t is not None else None for t in res]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,V", [(1, 8), (7, 1000), (33, 32000), (5, 128256), (300, 4096)])
def test_xent_shapes(rf, dtype, rows, V):
    logits, targets = inputs.xent_inputs(rows, V, dtype, seed=rows + V)
    targets[::3] = -100  # some ignored rows
    loss, lse, grad = run(rf, logits, targets)
    rloss, rlse, rgrad = oracle.softmax_xent(logits, targets)
    tol = 1e-5 * max(1.0, float(np.abs(rlse).max())) if dtype == "f32" else 1e-3
    assert np.abs(to64(lse) - rlse).max() <= tol
    assert np.abs(to64(loss) - rloss).max() <= tol
    assert (to64(loss)[::3] == 0).all() and (to64(grad)[::3] == 0).all()
    if dtype == "f32":
        assert np.abs(to64(grad) - rgrad).max() <= 1e-5
    else:
        assert np.abs(to64(grad) - rgrad).max() <= 2e-2  # grad rounded to 16 bits


def test_xent_out_of_range_target_gives_nan(rf):
    logits, targets = inputs.xent_inputs(4, 256, "bf16", seed=9)
    targets[1] = 256
    targets[2] = -7
    loss, lse = run(rf, logits, targets, want_grad=False)
    assert np.isnan(to64(loss)[[1, 2]]).all() and np.isfinite(to64(loss)[[0, 3]]).all()
    assert np.isfinite(to64(lse)).all()


def test_xent_large_logits(rf):
    logits, targets = inputs.xent_inputs(16, 4096, "f32", seed=10, scale=200.0)
    loss, lse, grad = run(rf, logits, targets)
    rloss, rlse, rgrad = oracle.softmax_xent(logits, targets)
    assert np.abs(to64(lse) - rlse).max() <= 1e-5 * np.abs(rlse).max()
    assert np.isfinite(to64(grad)).all()
    np.testing.assert_allclose(to64(grad).sum(-1), 0.0, atol=1e-4)


@pytest.mark.slow
def test_xent_full_size_sampled(rf):
    w = inputs.WORKLOADS["softmax_xent_bf16"]
    logits, targets = inputs.make(w)
    loss, lse = run(rf, logits, targets, want_grad=False)
    rows = np.unique(np.concatenate([[0, w.dims["rows"] - 1], np.random.default_rng(3).integers(0, w.dims["rows"], 62)]))
    rloss, rlse, _ = oracle.softmax_xent(logits[rows], targets[rows])
    assert np.abs(to64(lse)[rows] - rlse).max() <= 1e-3
    assert np.abs(to64(loss)[rows] - rloss).max() <= 1e-3


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,V", [(1, 128256), (2, 50000), (16, 128256), (64, 50000), (151, 32768), (152, 32768),
                                    (3, 16392)])
def test_xent_few_rows_cluster_path(rf, dtype, rows, V):
    """Few rows: each row is split over a cluster of up to 8 CTAs whose partial
    (max, sum exp) meet in distributed shared memory (ragged slices included)."""
    logits, targets = inputs.xent_inputs(rows, V, dtype, seed=rows * 7 + V)
    targets[::5] = -100
    bad = rows > 2  # row 1 gets a target outside [0, V): NaN loss, LSE still defined
    if bad:
        targets[1] = V + 3
    loss, lse, grad = run(rf, logits, targets)
    valid_t = targets.clone()
    if bad:
        valid_t[1] = -100  # the oracle takes targets in range or ignored only
    rloss, rlse, rgrad = oracle.softmax_xent(logits, valid_t)
    tol = 1e-5 * max(1.0, float(np.abs(rlse).max())) if dtype == "f32" else 1e-3
    assert np.abs(to64(lse) - rlse).max() <= tol
    keep = np.ones(rows, dtype=bool)
    if bad:
        keep[1] = False
        assert np.isnan(to64(loss)[1])
    assert np.abs(to64(loss)[keep] - rloss[keep]).max() <= tol
    assert (to64(grad)[::5] == 0).all()
    assert np.abs(to64(grad)[keep] - rgrad[keep]).max() <= (1e-5 if dtype == "f32" else 2e-2)
