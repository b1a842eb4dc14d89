"""ctypes binding of librf.so, the C ABI declared in include/rf.h.

Argument marshalling only: each ``rf_*`` function here takes torch tensors
that already live on the GPU, reads their shapes, pointers and dtype, and calls
the C function of the same name.  Every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if librf.so is missing the
first call raises, and a non-OK status raises ``RFError`` with the library's
message.

The ``attention``, ``decode`` and ``layernorm`` helpers additionally allocate
the outputs (and the decode workspace) with torch before calling the C ABI.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librf.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "rf.h")

RF_OK, RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_CUDA, RF_ERR_TIMEOUT, RF_ERR_CHECK = range(6)
STATUS_NAMES = {0: "RF_OK", 1: "RF_ERR_INVALID_ARG", 2: "RF_ERR_UNSUPPORTED", 3: "RF_ERR_CUDA", 4: "RF_ERR_TIMEOUT",
                5: "RF_ERR_CHECK"}
DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

_lib = None

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class AttnOpts(ctypes.Structure):
    """rf_attn_opts_t: causal mask, sliding window, ALiBi slopes (device fp32 [Hq]), split-tail workspace,
    rotary embedding inside the kernel (mode, base, position offset)."""
    _fields_ = [("causal", ctypes.c_int), ("window", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("rope", ctypes.c_int), ("rope_base", ctypes.c_float), ("rope_pos_offset", ctypes.c_int)]
_SIGNATURES = {
    "rf_attn_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "rf_attn_fwd_ex": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, ctypes.POINTER(AttnOpts), _i, _vp], _i),
    "rf_attn_fwd_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "rf_attn_decode_splitkv_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "rf_attn_decode_splitkv": ([_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "rf_attn_decode_splitkv_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp], _i),
    "rf_lse_merge": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "rf_layernorm_fused": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _vp], _i),
    "rf_rmsnorm_fused": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _vp], _i),
    "rf_softmax_xent": ([_vp, _vp, _vp, _vp, _vp, _i, _i, ctypes.c_longlong, _i, _vp], _i),
    "rf_last_error": ([], ctypes.c_char_p),
    "rf_version": ([], _i),
    "rf_device_status": ([_vp, _i], _i),
    "rf_selftest_wait_timeout": ([ctypes.c_uint, _vp], _i),
    "rf_selftest_check": ([_vp], _i),
    "rf_checks_enabled": ([], _i),
    "rf_ablation_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "rf_rope_qk": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "rf_layernorm_ablation": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _vp, _sz, _i, _vp], _i),
    "rf_softmax_xent_ablation": ([_vp, _vp, _vp, _vp, _i, _i, ctypes.c_longlong, _i, _vp, _sz, _i, _vp], _i),
}


class RFError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str | None = None):
    """Load librf.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("RF_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"librf.so not found at {path}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def declared_symbols(header: str = HEADER):
    """Names of the functions declared in include/rf.h."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rf_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != RF_OK:
        raise RFError(status, load().rf_last_error().decode())


def _dev(t, name, nullable=False):
    if t is None:
        if nullable:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _code(dtype):
    if dtype not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dtype}")
    return DTYPE_CODES[dtype]


def rf_version() -> int:
    return load().rf_version()


def rf_last_error() -> str:
    return load().rf_last_error().decode()


def rf_device_status(stream=None, clear=True) -> int:
    """Synchronise the stream and return the device status (RF_OK, RF_ERR_CHECK or RF_ERR_TIMEOUT)."""
    return load().rf_device_status(_stream(stream), int(bool(clear)))


def rf_selftest_wait_timeout(timeout_us=2000, stream=None):
    """Launch the bounded-wait self-test (a wait that is meant to run out)."""
    _check(load().rf_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def rf_selftest_check(stream=None):
    """Launch the index-check self-test (a check that always fails, no memory access)."""
    _check(load().rf_selftest_check(_stream(stream)))


def rf_checks_enabled() -> bool:
    """True for a library built with -DRF_CHECKS (every kernel checks its indices)."""
    return bool(load().rf_checks_enabled())


def rf_attn_fwd(q, k, v, o, lse=None, scale=None, causal=False, stream=None):
    """o[B,Hq,Nq,D] (and lse[B,Hq,Nq] fp32) <- attention(q[B,Hq,Nq,D], k/v[B,Hkv,Nk,D])."""
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, D) or tuple(v.shape) != tuple(k.shape) or tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch among q, k, v, o")
    if not (q.dtype == k.dtype == v.dtype == o.dtype):
        raise ValueError("q, k, v and o must share a dtype")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq)):
        raise ValueError("lse must be float32 [B,Hq,Nq]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().rf_attn_fwd(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _dev(lse, "lse", True),
                              B, Hq, Hkv, Nq, Nk, D, scale, int(bool(causal)), _code(q.dtype), _stream(stream)))


def rf_attn_fwd_ex(q, k, v, o, lse=None, scale=None, causal=False, window=0, alibi_slopes=None, workspace=None,
                   stream=None, rope=0, rope_base=10000.0, rope_pos_offset=0):
    """rf_attn_fwd with a sliding window (key j visible iff i - window < j <= i) and/or
    ALiBi slopes (float32 CUDA tensor [Hq]), both needing causal=True, an optional
    workspace (uint8 CUDA tensor, see attn_workspace) for splitting a short last wave,
    and rotary embedding inside the kernel (rope=1: Q rows, rope=2: Q and K rows)."""
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, D) or tuple(v.shape) != tuple(k.shape) or tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch among q, k, v, o")
    if not (q.dtype == k.dtype == v.dtype == o.dtype):
        raise ValueError("q, k, v and o must share a dtype")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq)):
        raise ValueError("lse must be float32 [B,Hq,Nq]")
    if alibi_slopes is not None and (alibi_slopes.dtype != torch.float32 or alibi_slopes.numel() != Hq):
        raise ValueError("alibi_slopes must be float32 with Hq elements")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = AttnOpts(int(bool(causal)), int(window), _dev(alibi_slopes, "alibi_slopes", True),
                    _dev(workspace, "workspace", True), wsb, int(rope), float(rope_base), int(rope_pos_offset))
    _check(load().rf_attn_fwd_ex(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _dev(lse, "lse", True),
                                 B, Hq, Hkv, Nq, Nk, D, scale, ctypes.byref(opts), _code(q.dtype), _stream(stream)))


def rf_attn_fwd_workspace_bytes(B, Hq, Nq, Nk, D, causal, dtype) -> int:
    """Workspace bytes rf_attn_fwd_ex can use on the current device (0: nothing to split)."""
    n = load().rf_attn_fwd_workspace_bytes(int(B), int(Hq), int(Nq), int(Nk), int(D), int(bool(causal)),
                                           _code(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise RFError(RF_ERR_INVALID_ARG, "rf_attn_fwd_workspace_bytes: invalid arguments or no device")
    return n


def attn_workspace(q, k, causal=False):
    """A uint8 workspace for rf_attn_fwd_ex's split tail, or None when nothing would be split."""
    B, Hq, Nq, D = q.shape
    n = rf_attn_fwd_workspace_bytes(B, Hq, Nq, k.shape[2], D, causal, q.dtype)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits) -> int:
    return load().rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits)


def rf_attn_decode_splitkv(q, k_cache, v_cache, o, workspace, num_splits, lse=None, scale=None, stream=None):
    """o[B,Hq,D] (and lse[B,Hq]) <- one-query attention over k/v_cache[B,Hkv,L,D], split in num_splits."""
    if q.dim() == 4:
        q = q.reshape(q.shape[0], q.shape[1], q.shape[3])
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, L, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shape mismatch")
    if o.numel() != B * Hq * D or o.dtype != q.dtype:
        raise ValueError("o must hold B*Hq*D elements of q's dtype")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != B * Hq):
        raise ValueError("lse must be float32 with B*Hq elements")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().rf_attn_decode_splitkv(_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                         _dev(o, "o"), _dev(lse, "lse", True), _dev(workspace, "workspace"),
                                         ws_bytes, B, Hq, Hkv, L, D, int(num_splits), scale, _code(q.dtype),
                                         _stream(stream)))


def rf_attn_decode_splitkv_noalloc(q, k_cache, v_cache, o, num_splits, lse=None, scale=None, stream=None):
    """rf_attn_decode_splitkv for callers that cannot allocate: the split partials go to
    scratch built into the library (RF_DECODE_NOALLOC_SCRATCH_BYTES), not to a workspace.
    Calls that may overlap on the GPU share that scratch and must be serialised."""
    if q.dim() == 4:
        q = q.reshape(q.shape[0], q.shape[1], q.shape[3])
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, L, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shape mismatch")
    if o.numel() != B * Hq * D or o.dtype != q.dtype:
        raise ValueError("o must hold B*Hq*D elements of q's dtype")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != B * Hq):
        raise ValueError("lse must be float32 with B*Hq elements")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().rf_attn_decode_splitkv_noalloc(_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                                 _dev(o, "o"), _dev(lse, "lse", True), B, Hq, Hkv, L, D,
                                                 int(num_splits), scale, _code(q.dtype), _stream(stream)))


def rf_lse_merge(o_part, lse_part, o, lse=None, stream=None):
    """o[rows,D] (and lse[rows]) <- merge of o_part[rows,S,D], lse_part[rows,S] (fp32)."""
    rows, S, D = o_part.shape
    if o_part.dtype != torch.float32 or lse_part.dtype != torch.float32 or tuple(lse_part.shape) != (rows, S):
        raise ValueError("o_part [rows,S,D] and lse_part [rows,S] must be float32")
    if o.numel() != rows * D:
        raise ValueError("o must hold rows*D elements")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != rows):
        raise ValueError("lse must be float32 with rows elements")
    _check(load().rf_lse_merge(_dev(o_part, "o_part"), _dev(lse_part, "lse_part"), _dev(o, "o"),
                               _dev(lse, "lse", True), rows, S, D, _code(o.dtype), _stream(stream)))


def rf_layernorm_fused(x, residual, gamma, beta, out, eps=1e-5, residual_out=None, stream=None):
    """out[rows,cols] <- LayerNorm(x + residual) * gamma + beta (residual/gamma/beta/residual_out may be None)."""
    rows, cols = x.shape
    for name, t in (("residual", residual), ("out", out), ("residual_out", residual_out)):
        if t is not None and (tuple(t.shape) != (rows, cols) or t.dtype != x.dtype):
            raise ValueError(f"{name} must match x")
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t is not None and (t.numel() != cols or t.dtype != x.dtype):
            raise ValueError(f"{name} must hold cols elements of x's dtype")
    _check(load().rf_layernorm_fused(_dev(x, "x"), _dev(residual, "residual", True), _dev(gamma, "gamma", True),
                                     _dev(beta, "beta", True), _dev(out, "out"),
                                     _dev(residual_out, "residual_out", True), rows, cols, float(eps),
                                     _code(x.dtype), _stream(stream)))


def rf_rmsnorm_fused(x, residual, gamma, out, eps=1e-5, residual_out=None, stream=None):
    """out[rows,cols] <- RMSNorm(x + residual) * gamma (residual/gamma/residual_out may be None)."""
    rows, cols = x.shape
    for name, t in (("residual", residual), ("out", out), ("residual_out", residual_out)):
        if t is not None and (tuple(t.shape) != (rows, cols) or t.dtype != x.dtype):
            raise ValueError(f"{name} must match x")
    if gamma is not None and (gamma.numel() != cols or gamma.dtype != x.dtype):
        raise ValueError("gamma must hold cols elements of x's dtype")
    _check(load().rf_rmsnorm_fused(_dev(x, "x"), _dev(residual, "residual", True), _dev(gamma, "gamma", True),
                                   _dev(out, "out"), _dev(residual_out, "residual_out", True), rows, cols,
                                   float(eps), _code(x.dtype), _stream(stream)))


def rf_softmax_xent(logits, targets, loss, lse=None, grad=None, ignore_index=-100, stream=None):
    """loss[rows] (and lse[rows], grad[rows,V]) <- cross-entropy of logits[rows,V] at int64 targets[rows]."""
    rows, V = logits.shape
    if targets.dtype != torch.int64 or targets.numel() != rows:
        raise ValueError("targets must be int64 with rows elements")
    if loss.dtype != torch.float32 or loss.numel() != rows:
        raise ValueError("loss must be float32 with rows elements")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != rows):
        raise ValueError("lse must be float32 with rows elements")
    if grad is not None and (tuple(grad.shape) != (rows, V) or grad.dtype != logits.dtype):
        raise ValueError("grad must match logits")
    _check(load().rf_softmax_xent(_dev(logits, "logits"), _dev(targets, "targets"), _dev(loss, "loss"),
                                  _dev(lse, "lse", True), _dev(grad, "grad", True), rows, V, int(ignore_index),
                                  _code(logits.dtype), _stream(stream)))


def alibi_slopes(n_heads, device="cuda"):
    """ALiBi head slopes, the geometric sequence 2^(-8 (h+1) / H), as float32 [H]."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / n_heads) for h in range(n_heads)], dtype=torch.float32,
                        device=device)


# ------------------------------------------------------------------ allocating helpers
def attention(q, k, v, scale=None, causal=False, window=0, alibi_slopes=None, split_tail=True, stream=None,
              rope=0, rope_base=10000.0, rope_pos_offset=0):
    """Allocate (o, lse) and run rf_attn_fwd_ex; with split_tail (the default) a short last
    wave of the unmasked 16-bit kernel is split along the keys (a workspace is allocated)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    ws = None
    if split_tail and not causal and q.dtype != torch.float32:
        ws = attn_workspace(q, k, causal)
    rf_attn_fwd_ex(q, k, v, o, lse, scale=scale, causal=causal, window=window, alibi_slopes=alibi_slopes,
                   workspace=ws, stream=stream, rope=rope, rope_base=rope_base, rope_pos_offset=rope_pos_offset)
    return o, lse


def decode_workspace(B, Hq, D, num_splits, device="cuda"):
    n = rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode(q, k_cache, v_cache, num_splits, scale=None, workspace=None, stream=None):
    """Allocate (o [B,Hq,D], lse [B,Hq]) and a workspace if none is given, then run rf_attn_decode_splitkv."""
    B, Hq, D = q.shape[0], q.shape[1], q.shape[-1]
    if workspace is None:
        workspace = decode_workspace(B, Hq, D, num_splits, q.device)
    o = torch.empty((B, Hq, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    rf_attn_decode_splitkv(q, k_cache, v_cache, o, workspace, num_splits, lse=lse, scale=scale, stream=stream)
    return o, lse


def decode_partials_view(workspace, B, Hq, D, num_splits):
    """(o_part [B,Hq,S,D], lse_part [B,Hq,S]) views of a decode workspace."""
    rows = B * Hq
    o_bytes = (rows * num_splits * D * 4 + 255) // 256 * 256
    o_part = workspace[: rows * num_splits * D * 4].view(torch.float32).view(B, Hq, num_splits, D)
    lse_part = workspace[o_bytes: o_bytes + rows * num_splits * 4].view(torch.float32).view(B, Hq, num_splits)
    return o_part, lse_part


def rmsnorm(x, residual, gamma, eps=1e-5, want_residual_out=False, stream=None):
    out = torch.empty_like(x)
    rout = torch.empty_like(x) if want_residual_out else None
    rf_rmsnorm_fused(x, residual, gamma, out, eps=eps, residual_out=rout, stream=stream)
    return (out, rout) if want_residual_out else out


def softmax_xent(logits, targets, ignore_index=-100, want_grad=False, stream=None):
    rows = logits.shape[0]
    loss = torch.empty(rows, dtype=torch.float32, device=logits.device)
    lse = torch.empty(rows, dtype=torch.float32, device=logits.device)
    grad = torch.empty_like(logits) if want_grad else None
    rf_softmax_xent(logits, targets, loss, lse, grad, ignore_index=ignore_index, stream=stream)
    return (loss, lse, grad) if want_grad else (loss, lse)


def layernorm(x, residual, gamma, beta, eps=1e-5, want_residual_out=False, stream=None):
    out = torch.empty_like(x)
    rout = torch.empty_like(x) if want_residual_out else None
    rf_layernorm_fused(x, residual, gamma, beta, out, eps=eps, residual_out=rout, stream=stream)
    return (out, rout) if want_residual_out else out


def rf_rope_qk(q, k=None, q_out=None, k_out=None, base=10000.0, pos_offset=0, stream=None):
    """Rotary embedding of q [B,Hq,N,D] (and k [B,Hkv,N,D]) at positions pos_offset + n; in place by default."""
    q_out = q if q_out is None else q_out
    k_out = k if k_out is None else k_out
    B, Hq, N, D = q.shape
    Hkv = 0
    if k is not None:
        if k.dim() != 4 or k.shape[0] != B or k.shape[2] != N or k.shape[3] != D or k.dtype != q.dtype:
            raise ValueError("k must be [B,Hkv,N,D] of q's dtype")
        Hkv = k.shape[1]
        if tuple(k_out.shape) != tuple(k.shape) or k_out.dtype != k.dtype:
            raise ValueError("k_out must match k")
    if tuple(q_out.shape) != tuple(q.shape) or q_out.dtype != q.dtype:
        raise ValueError("q_out must match q")
    _check(load().rf_rope_qk(_dev(q, "q"), _dev(k, "k", True), _dev(q_out, "q_out"), _dev(k_out, "k_out", True),
                             B, Hq, Hkv, N, D, float(base), int(pos_offset), _code(q.dtype), _stream(stream)))
    return q_out, k_out


LN_VARIANTS = {0: "fused incremental", 1: "fused non-incremental (row in shared memory)",
               2: "reductions fused, normalise separate", 3: "unfused"}
XENT_VARIANTS = {0: "fused incremental", 1: "fused two-pass", 2: "unfused"}


def rf_ablation_workspace_bytes(op, variant, rows, cols, dtype) -> int:
    """Workspace bytes of an ablation variant (op 0 = LayerNorm, 1 = cross-entropy)."""
    n = load().rf_ablation_workspace_bytes(int(op), int(variant), int(rows), int(cols), _code(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise RFError(RF_ERR_INVALID_ARG, "rf_ablation_workspace_bytes: invalid arguments")
    return n


def rf_layernorm_ablation(x, residual, gamma, beta, out, variant, workspace=None, eps=1e-5, stream=None):
    """LayerNorm(x + residual) * gamma + beta computed by ablation `variant` (see LN_VARIANTS)."""
    rows, cols = x.shape
    for name, t in (("residual", residual), ("out", out)):
        if t is None or tuple(t.shape) != (rows, cols) or t.dtype != x.dtype:
            raise ValueError(f"{name} must match x")
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t is None or t.numel() != cols or t.dtype != x.dtype:
            raise ValueError(f"{name} must hold cols elements of x's dtype")
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().rf_layernorm_ablation(_dev(x, "x"), _dev(residual, "residual"), _dev(gamma, "gamma"),
                                        _dev(beta, "beta"), _dev(out, "out"), rows, cols, float(eps), int(variant),
                                        _dev(workspace, "workspace", True), wsb, _code(x.dtype), _stream(stream)))


def rf_softmax_xent_ablation(logits, targets, loss, lse, variant, workspace=None, ignore_index=-100, stream=None):
    """Cross-entropy loss (and lse) computed by ablation `variant` (see XENT_VARIANTS)."""
    rows, V = logits.shape
    if targets.dtype != torch.int64 or targets.numel() != rows:
        raise ValueError("targets must be int64 with rows elements")
    for name, t in (("loss", loss), ("lse", lse)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != rows):
            raise ValueError(f"{name} must be float32 with rows elements")
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().rf_softmax_xent_ablation(_dev(logits, "logits"), _dev(targets, "targets"), _dev(loss, "loss"),
                                           _dev(lse, "lse", True), rows, V, int(ignore_index), int(variant),
                                           _dev(workspace, "workspace", True), wsb, _code(logits.dtype),
                                           _stream(stream)))


def ablation_workspace(op, variant, rows, cols, dtype, device="cuda"):
    """A device workspace (uint8) large enough for the variant, or None when it needs none."""
    n = rf_ablation_workspace_bytes(op, variant, rows, cols, dtype)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


__all__ = [
    "RFError", "load", "declared_symbols", "rf_version", "rf_last_error", "rf_device_status",
    "rf_selftest_wait_timeout", "rf_selftest_check", "rf_checks_enabled", "rf_attn_fwd",
    "rf_attn_fwd_ex", "AttnOpts", "alibi_slopes", "rf_attn_fwd_workspace_bytes", "attn_workspace",
    "rf_attn_decode_splitkv_workspace_bytes", "rf_attn_decode_splitkv", "rf_attn_decode_splitkv_noalloc",
    "rf_lse_merge", "rf_layernorm_fused", "rf_rmsnorm_fused", "rmsnorm", "rf_softmax_xent", "softmax_xent",
    "attention", "decode", "decode_workspace", "decode_partials_view", "layernorm",
    "rf_ablation_workspace_bytes", "rf_layernorm_ablation", "rf_softmax_xent_ablation", "ablation_workspace",
    "LN_VARIANTS", "XENT_VARIANTS", "rf_rope_qk",
    "RF_OK", "RF_ERR_INVALID_ARG", "RF_ERR_UNSUPPORTED", "RF_ERR_CUDA", "RF_ERR_TIMEOUT", "RF_ERR_CHECK",
    "STATUS_NAMES",
]
