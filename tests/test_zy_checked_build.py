"""The index-checked build (-DRF_CHECKS) on the GPU.

In that build every kernel checks the indices it computes (tensor coordinates,
output rows, split-tail and workspace slots, shared-memory tiles) and records
RF_ERR_CHECK in the device status word instead of making an access that falls
outside its buffer; nothing traps.  It stands in for a memory checker.  The
test builds it, then runs the small-shape GPU parity tests against it in a
child process (the conftest fixture there fails any test after which the
status word is not clean), and checks that the self-test of the check path
records RF_ERR_CHECK there and nothing in the regular build.  The file sorts
after every other GPU test file but the no-allocation one."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PARITY_FILES = ["test_gpu_attn_tc.py", "test_gpu_attn_f32.py", "test_gpu_attn_plain_entry.py",
                "test_gpu_attn_rope.py", "test_gpu_decode.py", "test_gpu_merge.py", "test_gpu_layernorm.py",
                "test_gpu_xent.py", "test_gpu_rope.py", "test_gpu_failure.py"]

CHILD_SELFTEST = """
import cascaded_reductions_pass_gb300 as rf
rf.load()
assert rf.rf_checks_enabled(), "not the checked build"
assert rf.rf_device_status() == rf.RF_OK
rf.rf_selftest_check()
assert rf.rf_device_status(clear=True) == rf.RF_ERR_CHECK
assert rf.rf_device_status() == rf.RF_OK
print("checked build: self-test ok")
"""


@pytest.fixture(scope="module")
def checked_lib():
    from cascaded_reductions_pass_gb300 import _build

    return _build.build(checks=True)


def _child(args, lib):
    env = dict(os.environ, RF_LIBRARY=lib)
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)


@pytest.mark.gpu
def test_check_selftest_records_nothing_in_the_regular_build(rf):
    assert not rf.rf_checks_enabled()
    rf.rf_selftest_check()
    assert rf.rf_device_status() == rf.RF_OK


@pytest.mark.gpu
def test_checked_build_selftest(rf, checked_lib):
    res = _child(["-c", CHILD_SELFTEST], checked_lib)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-2000:]


@pytest.mark.gpu
def test_checked_build_passes_small_parity_suite_with_clean_status(rf, checked_lib):
    files = [os.path.join("tests", f) for f in PARITY_FILES]
    res = _child(["-m", "pytest", *files, "-m", "gpu and not slow", "-x", "-q", "-p", "no:cacheprovider"],
                 checked_lib)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-2000:]
    assert " passed" in res.stdout
