"""Each planted mistake in the oracle must make its pin suite fail (CPU only).

This checks the pins themselves: a plausible slip anywhere in the oracle -- a
dropped scale or max, a wrong causal index, a wrong GQA head map, K used for V,
an exp with the wrong sign, overlapping splits, an unnormalised merge weight,
the unbiased variance, eps outside the square root, a dropped residual -- fails
at least one pin.
"""
import os
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import _oracle_mutants  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_attention.py", "tests/test_oracle_merge.py",
        "tests/test_oracle_layernorm.py", "tests/test_oracle_xent.py", "tests/test_oracle_rope.py",
        "tests/test_golden.py"]


@pytest.mark.parametrize("name", sorted(_oracle_mutants.MUTANTS))
def test_mutant_is_caught(name):
    env = dict(os.environ, RF_ORACLE_MUTANT=name)
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert "mutant" not in res.stderr or "found" not in res.stderr, res.stderr[-2000:]
    assert res.returncode == 1, f"mutant {name} survived the pins:\n{res.stdout[-1500:]}"
