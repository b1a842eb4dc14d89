"""rf_attn_decode_splitkv_noalloc: decoding for callers that cannot allocate.

Some callers cannot call cudaMalloc: a plugin whose host framework owns all
device memory and passes in only the inputs and outputs, or a serving loop that
reserves its memory at start-up and forbids allocation afterwards (an
allocation can synchronise the device and can fail under memory pressure in
the middle of a run).  This entry point gives them split-KV decoding with the
per-split partials kept in scratch built into the library.

The GPU test calls it through the C ABI twice in a row, on two different
problems, and checks each result against the workspace entry point's and
against the fp64 oracle, within the 16-bit tolerances used by every parity
test.  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import cascaded_reductions_pass_gb300 as rfmod
import oracle
from cascaded_reductions_pass_gb300 import inputs
from _parity import check16, check_lse

SCRATCH_BYTES = 16 << 20  # RF_DECODE_NOALLOC_SCRATCH_BYTES in include/rf.h


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from cascaded_reductions_pass_gb300 import _build

    _build.build()
    lib = rfmod.load()
    P = ctypes.c_void_p(0x10000)
    # 16 x 64 heads x 256 splits x 128 dims of fp32 partials = 128 MiB > 16 MiB
    assert lib.rf_attn_decode_splitkv_workspace_bytes(16, 64, 128, 256) > SCRATCH_BYTES
    st = lib.rf_attn_decode_splitkv_noalloc(P, P, P, P, None, 16, 64, 8, 4096, 128, 256, 0.1, 2, None)
    assert st == rfmod.RF_ERR_INVALID_ARG
    msg = lib.rf_last_error().decode()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(rf):
    cases = [
        # (B, Hq, Hkv, L, D, splits, dtype, seed); the first is the full 16-split
        # decoding geometry at a shorter cache, the second a different shape so the
        # scratch holds the first call's partials when the second starts.
        (16, 64, 8, 4096, 128, 16, "bf16", 31),
        (3, 24, 4, 1500, 64, 7, "f16", 32),
    ]
    for B, Hq, Hkv, L, D, S, dtype, seed in cases:
        q, k, v = (t.cuda() for t in inputs.decode_inputs(B, Hq, Hkv, L, D, dtype, seed))
        scale = float(np.float32(1 / np.sqrt(D)))
        o_ref, lse_ref = rf.decode(q, k, v, S, scale=scale)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(lse_ref)
        rf.rf_attn_decode_splitkv_noalloc(q, k, v, o, S, lse=lse, scale=scale)
        torch.cuda.synchronize()
        check16(o.cpu(), o_ref.float().cpu(), f"noalloc vs workspace ({B},{Hq},{L},{D},{S})")
        check_lse(lse.cpu(), lse_ref.cpu(), what="noalloc lse")
        ro, rl = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale)
        check16(o.cpu(), ro, f"noalloc vs oracle ({B},{Hq},{L},{D},{S})")
        check_lse(lse.cpu(), rl, what="noalloc lse vs oracle")
    assert rf.rf_device_status() == rf.RF_OK
