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


# A planted-mistake run of the oracle pin suite (see _oracle_mutants.py): the
# mutant is applied before any test module imports the oracle's functions.
if os.environ.get("RF_ORACLE_MUTANT"):
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import _oracle_mutants

    _oracle_mutants.apply(os.environ["RF_ORACLE_MUTANT"])
