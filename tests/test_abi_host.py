"""The C ABI on the host, without a GPU: librf.so loads, exports every function
that include/rf.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import subprocess

import pytest

import cascaded_reductions_pass_gb300 as rf
from cascaded_reductions_pass_gb300 import _binding


@pytest.fixture(scope="module")
def lib():
    from cascaded_reductions_pass_gb300 import _build

    _build.build()
    return rf.load()


def test_header_declares_the_four_calls():
    names = rf.declared_symbols()
    for n in ("rf_attn_fwd", "rf_attn_decode_splitkv", "rf_lse_merge", "rf_layernorm_fused",
              "rf_attn_decode_splitkv_workspace_bytes", "rf_last_error", "rf_version", "rf_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in rf.declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_regular_build_has_no_index_checks(lib):
    assert lib.rf_checks_enabled() == 0


def test_version(lib):
    assert lib.rf_version() == 10100  # 1.1.0: rotary embedding fields in rf_attn_opts_t


P = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: every case below fails a host check first
MIS = ctypes.c_void_p(0x10004)
S = ctypes.c_void_p(0)


def attn(lib, q=P, k=P, v=P, o=P, lse=None, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, D=64, scale=0.125, causal=0, dt=1):
    return lib.rf_attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dt, S)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(q=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(o=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(B=0), rf.RF_ERR_INVALID_ARG, "positive"),
    (dict(Nk=-1), rf.RF_ERR_INVALID_ARG, "positive"),
    (dict(Hq=3, Hkv=2), rf.RF_ERR_INVALID_ARG, "multiple"),
    (dict(scale=0.0), rf.RF_ERR_INVALID_ARG, "scale"),
    (dict(scale=float("nan")), rf.RF_ERR_INVALID_ARG, "scale"),
    (dict(dt=7), rf.RF_ERR_INVALID_ARG, "dtype"),
    (dict(k=MIS), rf.RF_ERR_INVALID_ARG, "aligned"),
    (dict(causal=1, Nq=8, Nk=9), rf.RF_ERR_UNSUPPORTED, "Nq == Nk"),
    (dict(D=96), rf.RF_ERR_UNSUPPORTED, "D in {64, 128}"),
    (dict(D=130, dt=0), rf.RF_ERR_UNSUPPORTED, "f32 path"),
    (dict(D=6, dt=0), rf.RF_ERR_UNSUPPORTED, "f32 path"),
])
def test_attn_rejects(lib, kw, status, msg):
    assert attn(lib, **kw) == status
    assert msg in lib.rf_last_error().decode()


def decode(lib, ws=P, ws_bytes=1 << 30, B=2, Hq=16, Hkv=2, L=100, D=128, S_=4, dt=2, q=P, o=P):
    return lib.rf_attn_decode_splitkv(q, P, P, o, None, ws, ws_bytes, B, Hq, Hkv, L, D, S_, 0.1, dt, S)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(ws=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(q=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(L=0), rf.RF_ERR_INVALID_ARG, "positive"),
    (dict(S_=0), rf.RF_ERR_INVALID_ARG, "positive"),
    (dict(Hq=15), rf.RF_ERR_INVALID_ARG, "multiple"),
    (dict(ws=ctypes.c_void_p(0x10010)), rf.RF_ERR_INVALID_ARG, "256-byte"),
    (dict(ws_bytes=100), rf.RF_ERR_INVALID_ARG, "too small"),
    (dict(dt=0), rf.RF_ERR_UNSUPPORTED, "f32"),
    (dict(D=96), rf.RF_ERR_UNSUPPORTED, "D must be"),
    (dict(Hq=32, Hkv=2), rf.RF_ERR_UNSUPPORTED, "at most 8"),
    (dict(S_=300), rf.RF_ERR_UNSUPPORTED, "256"),
])
def test_decode_rejects(lib, kw, status, msg):
    assert decode(lib, **kw) == status
    assert msg in lib.rf_last_error().decode()


def test_decode_workspace_size(lib):
    B, Hq, D, S_ = 16, 64, 128, 16
    n = lib.rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, S_)
    o_bytes = B * Hq * S_ * D * 4
    assert n == (o_bytes + 255) // 256 * 256 + B * Hq * S_ * 4
    assert lib.rf_attn_decode_splitkv_workspace_bytes(0, Hq, D, S_) == 0
    assert lib.rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, -1) == 0


@pytest.mark.parametrize("args,status,msg", [
    ((None, P, P, None, 4, 2, 8, 1), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, None, 0, 2, 8, 1), rf.RF_ERR_INVALID_ARG, "positive"),
    ((P, P, MIS, None, 4, 2, 8, 1), rf.RF_ERR_INVALID_ARG, "aligned"),
    ((P, P, P, None, 4, 2, 6, 1), rf.RF_ERR_UNSUPPORTED, "multiple of 4"),
    ((P, P, P, None, 4, 2, 516, 1), rf.RF_ERR_UNSUPPORTED, "multiple of 4"),
    ((P, P, P, None, 4, 257, 8, 1), rf.RF_ERR_UNSUPPORTED, "256"),
    ((P, P, P, None, 4, 2, 8, 9), rf.RF_ERR_INVALID_ARG, "dtype"),
])
def test_merge_rejects(lib, args, status, msg):
    assert lib.rf_lse_merge(*args, S) == status
    assert msg in lib.rf_last_error().decode()


@pytest.mark.parametrize("args,status,msg", [
    ((None, P, P, P, P, None, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, P, None, None, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, P, P, None, 0, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "positive"),
    ((P, P, P, P, P, None, 4, 64, -1.0, 2), rf.RF_ERR_INVALID_ARG, "eps"),
    ((P, P, P, P, P, MIS, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "aligned"),
    ((P, P, P, P, P, None, 4, 60, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "multiple of 8"),
    ((P, P, P, P, P, None, 4, 62, 1e-5, 0), rf.RF_ERR_INVALID_ARG, "multiple of 4"),
    ((P, P, P, P, P, None, 4, 32776, 1e-5, 1), rf.RF_ERR_UNSUPPORTED, "exceeds 32768"),
    ((P, P, P, P, P, None, 4, 16388, 1e-5, 0), rf.RF_ERR_UNSUPPORTED, "exceeds 16384"),
])
def test_layernorm_rejects(lib, args, status, msg):
    assert lib.rf_layernorm_fused(*args, S) == status
    assert msg in lib.rf_last_error().decode()


def test_binding_refuses_cpu_tensors(lib):
    import torch

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rf.rf_layernorm_fused(x, x, None, None, x)


@pytest.mark.parametrize("args,status,msg", [
    ((None, P, P, P, None, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, None, None, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, P, None, 4, 0, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "positive"),
    ((P, P, P, P, None, 4, 64, float("inf"), 2), rf.RF_ERR_INVALID_ARG, "eps"),
    ((P, MIS, P, P, None, 4, 64, 1e-5, 2), rf.RF_ERR_INVALID_ARG, "aligned"),
    ((P, P, P, P, None, 4, 20, 1e-5, 1), rf.RF_ERR_INVALID_ARG, "multiple of 8"),
    ((P, P, P, P, None, 4, 40000, 1e-5, 2), rf.RF_ERR_UNSUPPORTED, "exceeds"),
])
def test_rmsnorm_rejects(lib, args, status, msg):
    assert lib.rf_rmsnorm_fused(*args, S) == status
    assert msg in lib.rf_last_error().decode()


@pytest.mark.parametrize("args,status,msg", [
    ((None, P, P, None, None, 4, 64, -100, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, None, P, None, None, 4, 64, -100, 2), rf.RF_ERR_INVALID_ARG, "non-null"),
    ((P, P, P, None, None, 0, 64, -100, 2), rf.RF_ERR_INVALID_ARG, "positive"),
    ((P, P, P, None, MIS, 4, 64, -100, 2), rf.RF_ERR_INVALID_ARG, "aligned"),
    ((P, P, P, None, None, 4, 100, -100, 2), rf.RF_ERR_INVALID_ARG, "multiple of 8"),
    ((P, P, P, None, None, 4, 102, -100, 0), rf.RF_ERR_INVALID_ARG, "multiple of 4"),
    ((P, P, P, None, None, 4, 64, -100, 5), rf.RF_ERR_INVALID_ARG, "dtype"),
])
def test_softmax_xent_rejects(lib, args, status, msg):
    assert lib.rf_softmax_xent(*args, S) == status
    assert msg in lib.rf_last_error().decode()


def test_attn_ex_rejects(lib):
    from cascaded_reductions_pass_gb300._binding import AttnOpts

    def call(opts, **kw):
        a = dict(B=1, Hq=2, Hkv=1, Nq=8, Nk=8, D=64)
        a.update(kw)
        return lib.rf_attn_fwd_ex(P, P, P, P, None, a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["D"], 0.125,
                                  ctypes.byref(opts) if opts is not None else None, 1, S)

    assert call(AttnOpts(1, -1, None)) == rf.RF_ERR_INVALID_ARG and "window" in lib.rf_last_error().decode()
    assert call(AttnOpts(0, 16, None)) == rf.RF_ERR_UNSUPPORTED and "causal" in lib.rf_last_error().decode()
    assert call(AttnOpts(0, 0, 0x10000)) == rf.RF_ERR_UNSUPPORTED
    assert call(AttnOpts(1, 16, None), Nk=9) == rf.RF_ERR_UNSUPPORTED and "Nq == Nk" in lib.rf_last_error().decode()
    assert call(AttnOpts(1, 16, 0x10002)) == rf.RF_ERR_INVALID_ARG and "aligned" in lib.rf_last_error().decode()


def test_attn_ex_rejects_bad_rope_options(lib):
    from cascaded_reductions_pass_gb300._binding import AttnOpts

    def call(rope, base=0.0, pos=0, dtype=1, alibi=None, N=8):
        opts = AttnOpts(1, 0, alibi, None, 0, rope, base, pos)
        return lib.rf_attn_fwd_ex(P, P, P, P, None, 1, 2, 1, N, N, 64, 0.125, ctypes.byref(opts), dtype, S)

    err = lambda: lib.rf_last_error().decode()
    assert call(3) == rf.RF_ERR_INVALID_ARG and "rope" in err()
    assert call(-1) == rf.RF_ERR_INVALID_ARG and "rope" in err()
    assert call(1, pos=-5) == rf.RF_ERR_INVALID_ARG and "rope_pos_offset" in err()
    assert call(2, base=1.0) == rf.RF_ERR_INVALID_ARG and "rope_base" in err()
    assert call(2, base=-3.0) == rf.RF_ERR_INVALID_ARG and "rope_base" in err()
    assert call(2, base=float("inf")) == rf.RF_ERR_INVALID_ARG and "rope_base" in err()
    assert call(1, dtype=0) == rf.RF_ERR_UNSUPPORTED and "f16 or bf16" in err()
    assert call(1, alibi=0x10000) == rf.RF_ERR_UNSUPPORTED and "ALiBi" in err()
    assert call(2, pos=(1 << 24) - 4) == rf.RF_ERR_UNSUPPORTED and "2^24" in err()


def test_ablation_workspace_bytes(lib):
    f = lib.rf_ablation_workspace_bytes
    bad = ctypes.c_size_t(-1).value
    assert f(0, 0, 64, 4096, 2) == 0 and f(0, 1, 64, 4096, 2) == 0
    assert f(0, 2, 64, 4096, 2) == 64 * 8  # (mean, rstd) per row
    # mean + (mean, rstd) per row, rounded to 256 bytes, then h [rows, cols] in the input dtype
    assert f(0, 3, 64, 4096, 2) == 768 + 64 * 4096 * 2
    assert f(0, 3, 64, 4096, 0) == 768 + 64 * 4096 * 4
    assert f(1, 0, 16, 1024, 2) == 0 and f(1, 1, 16, 1024, 2) == 0 and f(1, 2, 16, 1024, 2) == 16 * 8
    for args in ((0, 4, 8, 8, 2), (1, 3, 8, 8, 2), (2, 0, 8, 8, 2), (0, 0, 0, 8, 2), (0, 0, 8, 8, 7)):
        assert f(*args) == bad


@pytest.mark.parametrize("kw, status, msg", [
    (dict(variant=4), rf.RF_ERR_INVALID_ARG, "variant"),
    (dict(variant=-1), rf.RF_ERR_INVALID_ARG, "variant"),
    (dict(residual=None), rf.RF_ERR_INVALID_ARG, "required"),
    (dict(beta=None), rf.RF_ERR_INVALID_ARG, "required"),
    (dict(variant=1, cols=56840), rf.RF_ERR_UNSUPPORTED, "shared-memory"),
    (dict(variant=2, ws=None), rf.RF_ERR_INVALID_ARG, "workspace"),
    (dict(variant=3, wsb=100), rf.RF_ERR_INVALID_ARG, "workspace"),
    (dict(variant=2, x=MIS), rf.RF_ERR_INVALID_ARG, "aligned"),
    (dict(variant=2, cols=12), rf.RF_ERR_INVALID_ARG, "multiple of 8"),
    (dict(variant=2, eps=-1.0), rf.RF_ERR_INVALID_ARG, "eps"),
    (dict(variant=0, cols=12), rf.RF_ERR_INVALID_ARG, "rf_layernorm_fused"),
])
def test_layernorm_ablation_rejects(lib, kw, status, msg):
    a = dict(x=P, residual=P, gamma=P, beta=P, out=P, rows=4, cols=64, eps=1e-5, variant=2, ws=P, wsb=1 << 20,
             dtype=2)
    a.update(kw)
    st = lib.rf_layernorm_ablation(a["x"], a["residual"], a["gamma"], a["beta"], a["out"], a["rows"], a["cols"],
                                   a["eps"], a["variant"], a["ws"], a["wsb"], a["dtype"], S)
    assert st == status
    assert msg in lib.rf_last_error().decode()


@pytest.mark.parametrize("kw, status, msg", [
    (dict(variant=3), rf.RF_ERR_INVALID_ARG, "variant"),
    (dict(variant=2, ws=None), rf.RF_ERR_INVALID_ARG, "workspace"),
    (dict(variant=2, wsb=8), rf.RF_ERR_INVALID_ARG, "workspace"),
    (dict(variant=1, logits=MIS), rf.RF_ERR_INVALID_ARG, "aligned"),
    (dict(variant=1, vocab=100), rf.RF_ERR_INVALID_ARG, "multiple of 8"),
    (dict(variant=1, loss=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(variant=0, rows=0), rf.RF_ERR_INVALID_ARG, "rf_softmax_xent"),
])
def test_softmax_xent_ablation_rejects(lib, kw, status, msg):
    a = dict(logits=P, targets=P, loss=P, lse=None, rows=4, vocab=64, variant=2, ws=P, wsb=1 << 20, dtype=2)
    a.update(kw)
    st = lib.rf_softmax_xent_ablation(a["logits"], a["targets"], a["loss"], a["lse"], a["rows"], a["vocab"], -100,
                                      a["variant"], a["ws"], a["wsb"], a["dtype"], S)
    assert st == status
    assert msg in lib.rf_last_error().decode()


def test_attn_workspace_bytes_host_cases(lib):
    f = lib.rf_attn_fwd_workspace_bytes
    bad = ctypes.c_size_t(-1).value
    assert f(1, 8, 1024, 1024, 64, 1, 1) == 0  # causal: never split
    assert f(1, 8, 1024, 1024, 64, 0, 0) == 0  # fp32 path: never split
    assert f(0, 8, 1024, 1024, 64, 0, 1) == bad
    assert f(1, 8, 1024, 1024, 96, 0, 1) == bad  # no tensor-core kernel for D=96
    assert f(1, 8, 1024, 1024, 64, 0, 9) == bad


def test_attn_ex_rejects_misaligned_workspace(lib):
    from cascaded_reductions_pass_gb300._binding import AttnOpts

    opts = AttnOpts(0, 0, None, 0x10008, 1 << 20)
    st = lib.rf_attn_fwd_ex(P, P, P, P, None, 1, 2, 1, 8, 8, 64, 0.125, ctypes.byref(opts), 1, S)
    assert st == rf.RF_ERR_INVALID_ARG and "aligned" in lib.rf_last_error().decode()


@pytest.mark.parametrize("kw, status, msg", [
    (dict(q=None), rf.RF_ERR_INVALID_ARG, "non-null"),
    (dict(k_out=None), rf.RF_ERR_INVALID_ARG, "both"),
    (dict(N=0), rf.RF_ERR_INVALID_ARG, "positive"),
    (dict(base=1.0), rf.RF_ERR_INVALID_ARG, "base"),
    (dict(base=-2.0), rf.RF_ERR_INVALID_ARG, "base"),
    (dict(pos_offset=-1), rf.RF_ERR_INVALID_ARG, "pos_offset"),
    (dict(q=MIS), rf.RF_ERR_INVALID_ARG, "aligned"),
    (dict(dtype=0), rf.RF_ERR_UNSUPPORTED, "fp32"),
    (dict(D=96), rf.RF_ERR_UNSUPPORTED, "D=96"),
    (dict(pos_offset=(1 << 24) - 4), rf.RF_ERR_UNSUPPORTED, "2^24"),
])
def test_rope_rejects(lib, kw, status, msg):
    a = dict(q=P, k=P, q_out=P, k_out=P, B=1, Hq=2, Hkv=1, N=8, D=64, base=10000.0, pos_offset=0, dtype=1)
    a.update(kw)
    st = lib.rf_rope_qk(a["q"], a["k"], a["q_out"], a["k_out"], a["B"], a["Hq"], a["Hkv"], a["N"], a["D"],
                        a["base"], a["pos_offset"], a["dtype"], S)
    assert st == status
    assert msg in lib.rf_last_error().decode()
