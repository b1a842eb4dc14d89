import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built librf.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of CPU or GPU time)")


@pytest.fixture(scope="session")
def rf():
    """The CUDA library binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cascaded_reductions_pass_gb300 as rfmod

    rfmod.load()  # raises loudly if librf.so is missing
    return rfmod


@pytest.fixture(autouse=True)
def _no_silent_timeout(request):
    """After every GPU test: no kernel may have recorded a bounded wait that ran
    out (RF_ERR_TIMEOUT in the device status word), or in a checked build a
    failed index check (RF_ERR_CHECK), without the test clearing it.  Results can still look right when a wait gives up in a CTA whose work
    was already done, so parity alone would not catch it."""
    yield
    if request.node.get_closest_marker("gpu") is None or "rf" not in request.fixturenames:
        return
    rfmod = request.getfixturevalue("rf")
    status = rfmod.rf_device_status(clear=True)
    assert status == rfmod.RF_OK, (f"a kernel recorded {rfmod.STATUS_NAMES.get(status, status)} "
                                   f"(a bounded wait that ran out, or a failed index check) during {request.node.nodeid}")


# A planted-mistake run of the oracle pin suite (see _oracle_mutants.py): the
# mutant is applied before any test module imports the oracle's functions.
if os.environ.get("RF_ORACLE_MUTANT"):
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import _oracle_mutants

    _oracle_mutants.apply(os.environ["RF_ORACLE_MUTANT"])
