"""Failure detection on the GPU without faulting or hanging it.

A device-side wait that runs out must record RF_ERR_TIMEOUT in the status word
and return, leaving the context usable: the self-test kernel waits on a barrier
that nothing signals, with a 2 ms limit.  The next calls still work."""
import numpy as np
import pytest
import torch

import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives(rf):
    assert rf.rf_device_status(clear=True) == rf.RF_OK
    rf.rf_selftest_wait_timeout(2000)
    assert rf.rf_device_status(clear=False) == rf.RF_ERR_TIMEOUT
    assert "bounded wait ran out" in rf.rf_last_error()
    assert rf.rf_device_status(clear=True) == rf.RF_ERR_TIMEOUT  # read, then cleared
    assert rf.rf_device_status(clear=True) == rf.RF_OK
    # the context is still usable: a real call runs and is correct
    x, r, g, b = inputs.ln_inputs(8, 1024, "bf16", seed=1)
    y = rf.layernorm(x.cuda(), r.cuda(), g.cuda(), b.cuda())
    torch.cuda.synchronize()
    check16(y.cpu(), oracle.layernorm(x, r, g, b, 1e-5)[0], "after timeout")
    assert rf.rf_device_status() == rf.RF_OK


def test_selftest_rejects_out_of_range_timeouts(rf):
    with pytest.raises(rf.RFError):
        rf.rf_selftest_wait_timeout(0)
    with pytest.raises(rf.RFError):
        rf.rf_selftest_wait_timeout(5_000_000)
