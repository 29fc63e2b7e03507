"""fp64 CPU oracle for the fused decoder operators -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never calls it.

It wraps ``oracle.c`` (plain single-threaded fp64 C, one loop per step of
each operator's definition) with ctypes.  Inputs are numpy arrays in their
storage type (float64, float32, or bfloat16 as uint16 bits) and are read by
the C code exactly as stored; results come back as float64 arrays.

Parity pins: see tests/test_oracle_pins.py.  Every function here is pinned by
closed forms, invariants, hand-worked values and central finite differences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_DT = {np.dtype(np.float64): 0, np.dtype(np.float32): 1, np.dtype(np.uint16): 2}
_P = ctypes.c_void_p
_I = ctypes.c_int64
_D = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc -O2, ISO C11: no FMA contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.orc_rmsnorm_fwd.argtypes = [_P, _P, ctypes.c_int, _I, _I, _D, _P, _P]
            lib.orc_rmsnorm_bwd.argtypes = [_P, _P, _P, ctypes.c_int, _I, _I, _D, _P, _P]
            lib.orc_rope.argtypes = [_P, ctypes.c_int, _P, _I, _I, _I, _I, _D, ctypes.c_int, _P]
            lib.orc_rope_ex.argtypes = [_P, ctypes.c_int, _P, _I, _I, _I, _I, _D, ctypes.c_int, ctypes.c_int, _P, _P,
                                        _I, _P]
            lib.orc_linear_swiglu_fwd.argtypes = [_P, _P, _P, ctypes.c_int, _I, _I, _I, _P]
            lib.orc_linear_swiglu_bwd.argtypes = [_P, _P, _P, _P, ctypes.c_int, _I, _I, _I, _P, _P, _P]
            lib.orc_rmsnorm_qkv_rope.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P, _I,
                                                 _I, _I, _I, _I, _I, _I, _D, _D, _P, _P, _P, _P]
            lib.orc_swiglu_fwd.argtypes = [_P, _P, ctypes.c_int, _I, _P]
            lib.orc_swiglu_bwd.argtypes = [_P, _P, _P, ctypes.c_int, _I, _P, _P]
            lib.orc_linear_ce.argtypes = [_P, _P, ctypes.c_int, _P, _I, _I, _I, _I, ctypes.c_int, _D,
                                          _P, _P, _P, _P]
            lib.orc_linear_ce_rows.argtypes = [_P, _P, ctypes.c_int, _P, _I, _I, _I, _I, ctypes.c_int, _D,
                                               _P, _I, _P, _P, _P]
            lib.orc_linear_ce_dw_rows.argtypes = [_P, _P, ctypes.c_int, _P, _I, _I, _I, _I, ctypes.c_int, _D,
                                                  _P, _P, _I, _P]
            for f in ("orc_rmsnorm_fwd", "orc_rmsnorm_bwd", "orc_rope", "orc_rope_ex", "orc_swiglu_fwd", "orc_swiglu_bwd", "orc_linear_swiglu_fwd",
                      "orc_linear_swiglu_bwd",
                      "orc_linear_ce", "orc_linear_ce_rows", "orc_linear_ce_dw_rows"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a):
    a = np.ascontiguousarray(a)
    return a, a.ctypes.data


def _dt(*arrs):
    dts = {a.dtype for a in arrs}
    if len(dts) != 1:
        raise TypeError(f"mixed input dtypes {dts}")
    return _DT[arrs[0].dtype]


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: oracle status {rc}")


def rmsnorm_fwd(x, w, eps):
    x, px = _c(x); w, pw = _c(w)
    rows, cols = x.shape[0] if x.ndim > 1 else 1, x.shape[-1]
    rows = x.size // cols
    y = np.empty(x.shape, np.float64); rstd = np.empty((rows,), np.float64)
    _check(_load().orc_rmsnorm_fwd(px, pw, _dt(x, w), rows, cols, eps, y.ctypes.data, rstd.ctypes.data),
           "rmsnorm_fwd")
    return y, rstd


def rmsnorm_bwd(dy, x, w, eps):
    dy, pdy = _c(dy); x, px = _c(x); w, pw = _c(w)
    cols = x.shape[-1]; rows = x.size // cols
    dx = np.empty(x.shape, np.float64); dw = np.empty((cols,), np.float64)
    _check(_load().orc_rmsnorm_bwd(pdy, px, pw, _dt(dy, x, w), rows, cols, eps, dx.ctypes.data, dw.ctypes.data),
           "rmsnorm_bwd")
    return dx, dw


def rope(t, theta, sign=1, pos=None):
    """t [B, S, NH, D]; pos [B, S] int32 or None (p = s)."""
    t, pt = _c(t)
    B, S, NH, D = t.shape
    ppos = None
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        assert pos.shape == (B, S)
        ppos = pos.ctypes.data
    out = np.empty(t.shape, np.float64)
    _check(_load().orc_rope(pt, _dt(t), ppos, B, S, NH, D, theta, int(sign), out.ctypes.data), "rope")
    return out


def rope_ex(t, theta=1e4, sign=1, pos=None, pairing="half", cos_tab=None, sin_tab=None):
    """RoPE variants on t [B, S, NH, D]: pairing "half" (i, i+D/2) or
    "interleaved" (2i, 2i+1); optional explicit cos/sin tables [n, D/2]."""
    t, pt = _c(t)
    B, S, NH, D = t.shape
    ppos = None
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        ppos = pos.ctypes.data
    pc = ps = None
    n_tab = 0
    if cos_tab is not None:
        cos_tab = np.ascontiguousarray(cos_tab, dtype=np.float64)
        sin_tab = np.ascontiguousarray(sin_tab, dtype=np.float64)
        assert cos_tab.shape == sin_tab.shape and cos_tab.shape[1] == D // 2
        pc, ps, n_tab = cos_tab.ctypes.data, sin_tab.ctypes.data, cos_tab.shape[0]
    out = np.empty(t.shape, np.float64)
    _check(_load().orc_rope_ex(pt, _dt(t), ppos, B, S, NH, D, float(theta), int(sign),
                               1 if pairing == "interleaved" else 0, pc, ps, n_tab, out.ctypes.data), "rope_ex")
    return out


def rmsnorm_qkv_rope(x, w, Wq, Wk, Wv, B, S, Hq, Hk, eps, theta=1e4, bq=None, bk=None, bv=None, pos=None,
                     cos_tab=None, sin_tab=None):
    """Fused RMSNorm + QKV projection (+ bias) + RoPE on q and k.
    x [B*S, H]; w [H]; Wq [Hq*D, H]; Wk, Wv [Hk*D, H]; optional biases; pos
    [B, S] int32; optional cos/sin tables [n, D/2] indexed by position.
    Returns q [B,S,Hq,D], k [B,S,Hk,D], v [B,S,Hk,D], rstd [B*S] in float64."""
    x, px = _c(x); w, pw = _c(w); Wq, pq = _c(Wq); Wk, pk = _c(Wk); Wv, pv = _c(Wv)
    H = x.shape[1]
    D = Wq.shape[0] // Hq if Hq else Wk.shape[0] // Hk
    arrs = [x, w, Wq, Wk, Wv]
    pb = []
    for b in (bq, bk, bv):
        if b is None:
            pb.append(None)
        else:
            b, p = _c(b)
            arrs.append(b)
            pb.append(p)
    ppos = None
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        ppos = pos.ctypes.data
    pc = ps = None
    n_tab = 0
    if cos_tab is not None:
        cos_tab = np.ascontiguousarray(cos_tab, dtype=np.float64)
        sin_tab = np.ascontiguousarray(sin_tab, dtype=np.float64)
        assert cos_tab.shape == sin_tab.shape and cos_tab.shape[1] == D // 2
        pc, ps, n_tab = cos_tab.ctypes.data, sin_tab.ctypes.data, cos_tab.shape[0]
    q = np.empty((B, S, Hq, D), np.float64)
    k = np.empty((B, S, Hk, D), np.float64)
    v = np.empty((B, S, Hk, D), np.float64)
    rstd = np.empty(B * S, np.float64)
    _check(_load().orc_rmsnorm_qkv_rope(px, pw, pq, pk, pv, pb[0], pb[1], pb[2], _dt(*arrs), ppos, pc, ps, n_tab,
                                        B, S, H, Hq, Hk, D, float(eps), float(theta), q.ctypes.data, k.ctypes.data,
                                        v.ctypes.data, rstd.ctypes.data), "rmsnorm_qkv_rope")
    return q, k, v, rstd


def swiglu_fwd(g, u):
    g, pg = _c(g); u, pu = _c(u)
    y = np.empty(g.shape, np.float64)
    _check(_load().orc_swiglu_fwd(pg, pu, _dt(g, u), g.size, y.ctypes.data), "swiglu_fwd")
    return y


def swiglu_bwd(dy, g, u):
    dy, pdy = _c(dy); g, pg = _c(g); u, pu = _c(u)
    dg = np.empty(g.shape, np.float64); du = np.empty(g.shape, np.float64)
    _check(_load().orc_swiglu_bwd(pdy, pg, pu, _dt(dy, g, u), g.size, dg.ctypes.data, du.ctypes.data),
           "swiglu_bwd")
    return dg, du


def linear_swiglu_fwd(X, Wg, Wu):
    """FusedLinearSwiGLU forward: silu(X Wg^T) * (X Wu^T)."""
    X, pX = _c(X); Wg, pg = _c(Wg); Wu, pu = _c(Wu)
    T, H = X.shape; I = Wg.shape[0]
    out = np.empty((T, I), np.float64)
    _check(_load().orc_linear_swiglu_fwd(pX, pg, pu, _dt(X, Wg, Wu), T, H, I, out.ctypes.data), "linear_swiglu_fwd")
    return out


def linear_swiglu_bwd(X, Wg, Wu, dH):
    """FusedLinearSwiGLU backward: (dX, dWg, dWu)."""
    X, pX = _c(X); Wg, pg = _c(Wg); Wu, pu = _c(Wu); dH, pd = _c(dH)
    T, H = X.shape; I = Wg.shape[0]
    dX = np.empty((T, H), np.float64); dWg = np.empty((I, H), np.float64); dWu = np.empty((I, H), np.float64)
    _check(_load().orc_linear_swiglu_bwd(pX, pg, pu, pd, _dt(X, Wg, Wu, dH), T, H, I, dX.ctypes.data,
                                         dWg.ctypes.data, dWu.ctypes.data), "linear_swiglu_bwd")
    return dX, dWg, dWu


def linear_ce(X, W, labels, ignore_index=-100, reduction="mean", grad_scale=1.0, want_grads=True):
    """Returns dict(loss, lse[T], dX[T,H], dW[V,H]) in float64."""
    X, pX = _c(X); W, pW = _c(W)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    T, H = X.shape; V = W.shape[0]
    assert W.shape[1] == H and labels.shape == (T,)
    loss = np.zeros((1,), np.float64); lse = np.empty((T,), np.float64)
    dX = np.empty((T, H), np.float64) if want_grads else None
    dW = np.empty((V, H), np.float64) if want_grads else None
    rc = _load().orc_linear_ce(pX, pW, _dt(X, W), labels.ctypes.data, T, H, V, int(ignore_index),
                               0 if reduction == "mean" else 1, float(grad_scale), loss.ctypes.data,
                               lse.ctypes.data, dX.ctypes.data if want_grads else None,
                               dW.ctypes.data if want_grads else None)
    _check(rc, "linear_ce")
    return {"loss": float(loss[0]), "lse": lse, "dX": dX, "dW": dW}


def linear_ce_rows(X, W, labels, rows, ignore_index=-100, reduction="mean", grad_scale=1.0):
    """The definition on selected rows: dict(lse[k], loss_term[k], dX[k, H])."""
    X, pX = _c(X); W, pW = _c(W)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    T, H = X.shape; V = W.shape[0]
    k = rows.size
    lse = np.empty((k,), np.float64); lt = np.empty((k,), np.float64); dX = np.empty((k, H), np.float64)
    rc = _load().orc_linear_ce_rows(pX, pW, _dt(X, W), labels.ctypes.data, T, H, V, int(ignore_index),
                                    0 if reduction == "mean" else 1, float(grad_scale), rows.ctypes.data, k,
                                    lse.ctypes.data, lt.ctypes.data, dX.ctypes.data)
    _check(rc, "linear_ce_rows")
    return {"lse": lse, "loss_term": lt, "dX": dX}


def linear_ce_rows_fwd(X, W, labels, rows, ignore_index=-100):
    """lse and the loss term (lse - z_label, 0 if ignored) of the listed rows, without dX."""
    X, pX = _c(X); W, pW = _c(W)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    T, H = X.shape; V = W.shape[0]
    k = rows.size
    lse = np.empty((k,), np.float64); lt = np.empty((k,), np.float64)
    rc = _load().orc_linear_ce_rows(pX, pW, _dt(X, W), labels.ctypes.data, T, H, V, int(ignore_index), 0, 1.0,
                                    rows.ctypes.data, k, lse.ctypes.data, lt.ctypes.data, None)
    _check(rc, "linear_ce_rows_fwd")
    return {"lse": lse, "loss_term": lt}


def linear_ce_dw_rows(X, W, labels, lse, vrows, ignore_index=-100, reduction="mean", grad_scale=1.0):
    """dW rows of the listed vocabulary rows, given lse [T] of every token."""
    X, pX = _c(X); W, pW = _c(W)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    vrows = np.ascontiguousarray(vrows, dtype=np.int64)
    T, H = X.shape; V = W.shape[0]
    out = np.empty((vrows.size, H), np.float64)
    rc = _load().orc_linear_ce_dw_rows(pX, pW, _dt(X, W), labels.ctypes.data, T, H, V, int(ignore_index),
                                       0 if reduction == "mean" else 1, float(grad_scale), lse.ctypes.data,
                                       vrows.ctypes.data, vrows.size, out.ctypes.data)
    _check(rc, "linear_ce_dw_rows")
    return out


def rel_err(got, ref):
    """max_i |g_i - o_i| / max(|o_i|, rms(o)) over one tensor (float64)."""
    got = np.asarray(got, np.float64).ravel(); ref = np.asarray(ref, np.float64).ravel()
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(got - ref) / den))
