"""Oracle: plain, slow, unfused CPU implementation of the cascaded reductions.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
anything from this package.  The CUDA library never calls it, and it shares no
code, header, table or constant with the CUDA path: both sides only consume the
same seeded inputs.

Everything here is numpy float64 and follows the plain definitions of the
operations, one whole-array pass per level of the cascade, never the fused or
incremental form that the CUDA kernels use:

* ``attention``     -- safe softmax followed by the GEMM (RedFuser, Abstract;
  "Operator Fusion" guide, section 2, Pattern 4 "Attention Fusion", the
  unfused listing): scores, optional causal mask, row max, exp, row sum,
  weighted sum of V, normalisation; plus the natural-log LSE per row.
* ``decode``        -- the same definition with one query per head over a KV
  cache (AttnFuse, Table 8 "Flash Decoding"; RedFuser, Figure 13
  "FlashDecoding IR").
* ``split_bounds`` / ``decode_partials`` -- attention restricted to contiguous
  key ranges, the per-split partial results that split-KV decoding combines.
* ``lse_merge``     -- the combine of partial results: LSE = ln sum_s exp(lse_s),
  O = sum_s exp(lse_s - LSE) O_s.
* ``layernorm``     -- residual add then mean -> biased variance -> normalise
  and affine ("Operator Fusion" guide, section 2, Pattern 2 "Reduction +
  Element-wise"; section 4 "Manual (CUDA)").
* ``rmsnorm``       -- residual add then mean of squares -> normalise and scale
  ("Operator Fusion" guide, section 3, fusible patterns: RMSNorm).
* ``softmax_xent``  -- row max -> sum exp -> cross-entropy loss, its LSE and
  gradient ("Operator Fusion" guide, section 3: softmax + cross-entropy).
* ``rope``          -- rotary position embedding of Q and K rows, the
  pre-matmul transformation of AttnFuse (Abstract; Figure 1), rotate-half
  pairing.

Every function is pinned by the CPU tests (brute force on tiny inputs, closed
forms, invariants, a library second opinion); no function is "parity unpinned".
"""
from .reference import (  # noqa: F401
    alibi_slopes,
    attention,
    decode,
    decode_partials,
    layernorm,
    lse_merge,
    rmsnorm,
    rope,
    softmax_xent,
    split_bounds,
)
