"""The C-ABI library: it loads, exports every function include/liger.h
declares, and rejects bad arguments on the host with the documented status
codes before touching the GPU (these calls make no CUDA call, so they run
without a GPU)."""
import ctypes
import os

import pytest

from transformer_rmsnorm_fwd_gb300 import _native


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        from transformer_rmsnorm_fwd_gb300 import build
        build.build()
    return _native.load()


def test_exports_every_declared_function(lib):
    names = _native.header_functions()
    assert len(names) == 26
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_native.SIGNATURES)


def test_status_codes_match_header():
    with open(_native.HEADER) as f:
        text = f.read()
    for code, name in _native.STATUS.items():
        if code:
            assert f"#define {name} ({code})" in text


def _err(lib):
    return lib.liger_last_error().decode()


def test_null_and_shape_errors(lib):
    assert lib.liger_rmsnorm_fwd(None, None, None, None, 4, 8, 1e-6, 0, None) == -1
    assert "required" in _err(lib)
    assert lib.liger_rmsnorm_fwd(None, None, None, None, -1, 8, 1e-6, 0, None) == -2
    assert lib.liger_rmsnorm_fwd(None, None, None, None, 4, 8, 1e-6, 7, None) == -3
    assert lib.liger_swiglu_fwd(None, None, None, 10, 1, None) == -1
    assert lib.liger_swiglu_fwd(None, None, None, -3, 1, None) == -2
    assert lib.liger_rope_fwd(None, None, None, 1, 4, 2, 2, 63, 1e4, 1, None) == -2      # odd head_dim
    assert lib.liger_rope_fwd(None, None, None, 1, 4, 2, 2, 64, -1.0, 1, None) == -2     # theta <= 0
    assert lib.liger_rope_fwd(None, None, None, 1, 4, 2, 2, 64, 1e4, 1, None) == -1
    assert lib.liger_linear_ce_fwd_bwd(None, None, None, 4, 8, 16, -100, 0, 1.0, None, None, None, None, 0, 0, 1,
                                       None) == -1
    assert lib.liger_linear_ce_fwd_bwd(None, None, None, 4, 8, 16, -100, 2, 1.0, None, None, None, None, 0, 0, 1,
                                       None) == -2


def test_alignment_and_workspace_errors(lib):
    bad = ctypes.c_void_p(0x1008)    # 8-byte aligned only, never dereferenced
    ok = ctypes.c_void_p(0x1000)
    assert lib.liger_swiglu_fwd(bad, ok, ok, 10, 1, None) == -4
    assert lib.liger_rmsnorm_fwd(ok, bad, ok, None, 4, 8, 1e-6, 1, None) == -4
    # workspace checks happen before any device work
    need = lib.liger_rmsnorm_bwd_workspace(4, 8)
    assert need == 4 * 8 * 4
    assert lib.liger_rmsnorm_bwd(ok, ok, ok, ok, ok, ok, ok, need - 1, 4, 8, 1, None) == -6
    n = lib.liger_linear_ce_workspace(100, 64, 1000, 0, 1)
    assert n > 0
    assert lib.liger_linear_ce_fwd_bwd(ok, ok, ok, 100, 64, 1000, -100, 0, 1.0, ok, None, None, ok, n - 1, 0, 1,
                                       None) == -6
    assert lib.liger_linear_ce_fwd_bwd(ok, ok, ok, 100, 64, 1000, -100, 0, 1.0, ok, None, None, ctypes.c_void_p(0x1010),
                                       n, 0, 1, None) == -6   # not 256-byte aligned
    # the forms without the host wait check their arguments the same way, before queueing anything
    for fn in (lib.liger_linear_ce_fwd_bwd_async, lib.liger_linear_ce_two_pass_fwd_bwd_async):
        assert fn(None, None, None, 4, 64, 256, -100, 0, 1.0, None, None, None, None, 0, 0, 1, None) == -1
        assert fn(ok, ok, ok, 4, 64, 256, -100, 2, 1.0, ok, None, None, ok, 1 << 30, 0, 1, None) == -2
        assert fn(ok, ok, ok, 100, 64, 1000, -100, 0, 1.0, ok, None, None, ok, 256, 0, 1, None) == -6
        assert fn(ok, ok, ok, 100, 64, 1000, -100, 0, 1.0, ok, None, None, ok, 1 << 30, 0, 7, None) == -3


def test_workspace_sizes(lib):
    # rmsnorm: min(rows, 1024) fp32 partial rows
    assert lib.liger_rmsnorm_bwd_workspace(32768, 4096) == 1024 * 4096 * 4
    assert lib.liger_rmsnorm_bwd_workspace(0, 4096) == 0
    # linear CE: never a [T x V] buffer -- at T=8192, V=128256 the chunk buffer is <= 4096 rows
    T, H, V = 8192, 4096, 128256
    n = lib.liger_linear_ce_workspace(T, H, V, 0, 1)
    full_logits = T * V * 2
    assert n < full_logits + V * H * 4
    assert lib.liger_linear_ce_workspace(T, H, V, 0, 7) == 0


def test_rmsnorm_qkv_rope_host_checks(lib):
    ok = ctypes.c_void_p(0x1000)
    r256 = lambda b: (b + 255) // 256 * 256
    T, H, Hq, Hk, D = 300, 320, 4, 2, 64
    N = (Hq + 2 * Hk) * D
    need = lib.liger_rmsnorm_qkv_rope_workspace(T, H, Hq, Hk, D)
    assert need == r256(N * H * 2) + r256(N * 4) + r256(T * 4) + 2 * r256(T * (D // 2) * 4)
    args = lambda **kw: [kw.get("x", ok), ok, ok, ok, ok, None, None, None, None, None, None, 0, ok, ok, ok, None,
                         kw.get("ws", ok), kw.get("ws_bytes", need), 2, 150, kw.get("H", H), Hq, Hk,
                         kw.get("D", D), 1e-6, kw.get("theta", 1e4), kw.get("flags", 0), kw.get("dtype", 1), None]
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(dtype=0)) == -3                 # fp32: tensor-core path is bf16
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(D=96)) == -2                    # head_dim not 64/128/256
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(H=324)) == -2                   # hidden not a multiple of 8
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(theta=0.0)) == -2
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(flags=2)) == -2
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(ws_bytes=need - 1)) == -6
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(ws=ctypes.c_void_p(0x1010))) == -6
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(x=None)) == -1
    assert lib.liger_rmsnorm_qkv_rope_fwd(*args(x=ctypes.c_void_p(0x1008))) == -4


def test_device_status_marker_checks_its_family(lib):
    # an unknown family is rejected before any CUDA call
    assert lib.liger_device_status_mark(4, None) == -2
    assert lib.liger_device_status_mark(-1, None) == -2
    assert "which" in _err(lib)
