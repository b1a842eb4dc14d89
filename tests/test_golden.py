"""Golden fixtures (CPU only).

* Values the pages print: the residual + LayerNorm traffic example of the
  "Operator Fusion" guide (section 1) pins the byte model used for roofline
  figures; RedFuser's Table 1 operator pairs pin the reduce/combine algebra.
* Values written by tests/golden/make_golden.py, which calls only the oracle:
  recomputing them guards the oracle against silent changes.
"""
import json
import os

import numpy as np
import pytest

import oracle
from cascaded_reductions_pass_gb300 import workmodel

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def dec(rec):
    """Decode a stored array to float64 (16-bit floats are widened exactly)."""
    raw = bytes.fromhex(rec["hex"])
    if rec["dtype"] == "f64":
        return np.frombuffer(raw, dtype=np.float64).reshape(rec["shape"])
    if rec["dtype"] == "f32":
        return np.frombuffer(raw, dtype=np.float32).reshape(rec["shape"]).astype(np.float64)
    if rec["dtype"] == "f16":
        return np.frombuffer(raw, dtype=np.float16).reshape(rec["shape"]).astype(np.float64)
    if rec["dtype"] == "bf16":
        u = np.frombuffer(raw, dtype=np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).reshape(rec["shape"]).astype(np.float64)
    raise ValueError(rec["dtype"])


def test_ln_traffic_matches_operator_fusion_page():
    g = load("operator_fusion_ln_traffic.json")
    rows, cols = g["B"] * g["S"], g["d"]
    tensor = rows * cols * workmodel.ELEM_BYTES[g["dtype"]]
    assert tensor == g["tensor_MiB"] * 2 ** 20
    fused = workmodel.layernorm_bytes(rows, cols, g["dtype"], affine=False)
    assert fused == (g["fused_reads"] + g["fused_writes"]) * tensor == g["fused_MiB"] * 2 ** 20


OPS = {"max": np.maximum, "min": np.minimum, "+": np.add, "*": np.multiply}


def test_table1_combine_distributes_over_reduce():
    rng = np.random.default_rng(0)
    a, b, c = rng.standard_normal((3, 512))
    for row in load("redfuser_table1_operator_pairs.json")["rows"]:
        red, comb = OPS[row["reduce"]], OPS[row["combine"]]
        # (a reduce b) combine c == (a combine c) reduce (b combine c)
        np.testing.assert_allclose(comb(red(a, b), c), red(comb(a, c), comb(b, c)), atol=1e-12,
                                   err_msg=row["reduction"])


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_oracle_reproduces_stored_fixtures():
    g = load("attn_small_oracle.json")
    q, k, v = dec(g["q"]), dec(g["k"]), dec(g["v"])
    for causal in (0, 1):
        o, lse = oracle.attention(q, k, v, g["scale"], bool(causal))
        np.testing.assert_allclose(o, dec(g[f"o_causal{causal}"]), atol=1e-12)
        np.testing.assert_allclose(lse, dec(g[f"lse_causal{causal}"]), atol=1e-12)
    g = load("decode_small_oracle.json")
    q, k, v = dec(g["q"]), dec(g["k"]), dec(g["v"])
    o, lse = oracle.decode(q, k, v, g["scale"])
    np.testing.assert_allclose(o, dec(g["o"]), atol=1e-12)
    np.testing.assert_allclose(lse, dec(g["lse"]), atol=1e-12)
    op, lp = oracle.decode_partials(q, k, v, g["scale"], g["num_splits"])
    np.testing.assert_allclose(op, dec(g["o_part"]), atol=1e-12)
    np.testing.assert_allclose(lp, dec(g["lse_part"]), atol=1e-12)
    g = load("merge_small_oracle.json")
    o, lse = oracle.lse_merge(dec(g["o_part"]), dec(g["lse_part"]))
    np.testing.assert_allclose(o, dec(g["o"]), atol=1e-12)
    np.testing.assert_allclose(lse, dec(g["lse"]), atol=1e-12)
    g = load("layernorm_small_oracle.json")
    y, h = oracle.layernorm(dec(g["x"]), dec(g["r"]), dec(g["gamma"]), dec(g["beta"]), g["eps"])
    np.testing.assert_allclose(y, dec(g["y"]), atol=1e-12)
    np.testing.assert_allclose(h, dec(g["h"]), atol=0)
