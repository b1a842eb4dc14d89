"""Write the oracle-computed golden fixtures of this folder.

Calls only the oracle (and the seeded input generator).  Inputs are stored
bit-exactly as hex so the fixtures do not depend on the random generator of a
particular torch version; outputs are stored as float64 hex.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from cascaded_reductions_pass_gb300 import inputs  # noqa: E402

BITS = {torch.float16: ("f16", np.uint16), torch.bfloat16: ("bf16", np.uint16), torch.float32: ("f32", np.uint32)}


def enc(t):
    name, it = BITS[t.dtype]
    bits = t.contiguous().view(torch.int16 if it is np.uint16 else torch.int32).numpy().astype(it)
    return {"dtype": name, "shape": list(t.shape), "hex": bits.tobytes().hex()}


def enc64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return {"dtype": "f64", "shape": list(a.shape), "hex": a.tobytes().hex()}


def dump(name, obj):
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(obj, f, indent=1)
        f.write("\n")


def main():
    # attention: fp16, GQA 2q/1kv, N = 12 (one ragged tile), D = 64; both masks
    q, k, v = inputs.attn_inputs(1, 2, 1, 12, 12, 64, "f16", seed=100)
    scale = float(np.float32(0.125))
    rec = {"about": "oracle attention on stored fp16 inputs; scale 0.125",
           "scale": scale, "q": enc(q), "k": enc(k), "v": enc(v)}
    for causal in (0, 1):
        o, lse = oracle.attention(q, k, v, scale, bool(causal))
        rec[f"o_causal{causal}"] = enc64(o)
        rec[f"lse_causal{causal}"] = enc64(lse)
    dump("attn_small_oracle.json", rec)

    # decode: bf16, 8 query heads on 1 kv head, L = 40 keys, D = 128, 3 splits
    q, k, v = inputs.decode_inputs(1, 8, 1, 40, 128, "bf16", seed=101)
    scale = float(np.float32(1.0 / np.sqrt(128.0)))
    o, lse = oracle.decode(q, k, v, scale)
    op, lp = oracle.decode_partials(q, k, v, scale, 3)
    dump("decode_small_oracle.json", {
        "about": "oracle decode (unsplit) and its 3 contiguous-split partials on stored bf16 inputs",
        "scale": scale, "num_splits": 3, "q": enc(q), "k": enc(k), "v": enc(v),
        "o": enc64(o), "lse": enc64(lse), "o_part": enc64(op), "lse_part": enc64(lp)})

    # merge: fp32 partials with empty splits
    o_part, lse_part = inputs.merge_inputs(4, 5, 8, seed=102, empty_frac=0.3)
    o, lse = oracle.lse_merge(o_part, lse_part)
    dump("merge_small_oracle.json", {
        "about": "oracle log-sum-exp merge of 5 fp32 partials per row, some empty (lse=-inf)",
        "o_part": enc(o_part), "lse_part": enc(lse_part), "o": enc64(o), "lse": enc64(lse)})

    # layernorm: bf16, 3 rows x 64 cols, eps 1e-5
    x, r, g, b = inputs.ln_inputs(3, 64, "bf16", seed=103)
    y, h = oracle.layernorm(x, r, g, b, 1e-5)
    dump("layernorm_small_oracle.json", {
        "about": "oracle residual+LayerNorm on stored bf16 inputs, eps 1e-5",
        "eps": 1e-5, "x": enc(x), "r": enc(r), "gamma": enc(g), "beta": enc(b),
        "y": enc64(y), "h": enc64(h)})


if __name__ == "__main__":
    main()
