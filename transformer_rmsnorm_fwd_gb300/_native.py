"""Thin Python binding of libliger.so (argument marshalling only).

Every function below has the name of the C entry point it calls and takes
torch tensors that already live on the GPU; it passes their device
pointers, sizes and the current CUDA stream to the library and raises
``LigerError`` on a non-zero status.  All computation happens in the
library's CUDA kernels; there is no fallback of any kind: if the library is
missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libliger.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "liger.h")

LIGER_F32, LIGER_BF16 = 0, 1
STATUS = {0: "OK", -1: "LIGER_ERR_NULL", -2: "LIGER_ERR_SHAPE", -3: "LIGER_ERR_DTYPE", -4: "LIGER_ERR_ALIGN",
          -5: "LIGER_ERR_LABEL", -6: "LIGER_ERR_WORKSPACE", -7: "LIGER_ERR_CUDA"}

_lib = None
_lock = threading.Lock()

_P, _I64, _F, _D, _INT, _SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_int,
                               ctypes.c_size_t)
SIGNATURES = {
    "liger_last_error": ([], ctypes.c_char_p),
    "liger_device_status": ([_P], _INT),
    "liger_device_status_mark": ([_INT, _P], _INT),
    "liger_rmsnorm_fwd": ([_P, _P, _P, _P, _I64, _I64, _F, _INT, _P], _INT),
    "liger_rmsnorm_bwd_workspace": ([_I64, _I64], _SZ),
    "liger_rmsnorm_bwd": ([_P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _INT, _P], _INT),
    "liger_rmsnorm_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "liger_rope_fwd": ([_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _D, _INT, _P], _INT),
    "liger_rope_bwd": ([_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _D, _INT, _P], _INT),
    "liger_rope_fwd_ex": ([_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P, _I64, _D, _INT, _P],
                          _INT),
    "liger_rope_bwd_ex": ([_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P, _I64, _D, _INT, _P],
                          _INT),
    "liger_swiglu_fwd": ([_P, _P, _P, _I64, _INT, _P], _INT),
    "liger_swiglu_bwd": ([_P, _P, _P, _P, _P, _I64, _INT, _P], _INT),
    "liger_fused_linear_swiglu_fwd": ([_P, _P, _P, _P, _I64, _I64, _I64, _INT, _P], _INT),
    "liger_fused_linear_swiglu_workspace": ([_I64, _I64], _SZ),
    "liger_fused_linear_swiglu_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _INT, _P], _INT),
    "liger_fused_linear_swiglu_fwd_save": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P], _INT),
    "liger_fused_linear_swiglu_bwd_saved": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I64, _I64, _INT, _P],
                                            _INT),
    "liger_rmsnorm_qkv_rope_workspace": ([_I64, _I64, _I64, _I64, _I64], _SZ),
    "liger_rmsnorm_qkv_rope_fwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _P, _SZ, _I64,
                                    _I64, _I64, _I64, _I64, _I64, _D, _D, _INT, _INT, _P], _INT),
    "liger_linear_ce_two_pass_workspace": ([_I64, _I64, _I64, _I64], _SZ),
    "liger_linear_ce_two_pass_fwd_bwd": ([_P, _P, _P, _I64, _I64, _I64, _I64, _INT, _F, _P, _P, _P, _P, _SZ, _I64,
                                          _INT, _P], _INT),
    "liger_linear_ce_workspace": ([_I64, _I64, _I64, _I64, _INT], _SZ),
    "liger_linear_ce_fwd_bwd": ([_P, _P, _P, _I64, _I64, _I64, _I64, _INT, _F, _P, _P, _P, _P, _SZ, _I64, _INT, _P],
                                _INT),
    "liger_linear_ce_fwd_bwd_async": ([_P, _P, _P, _I64, _I64, _I64, _I64, _INT, _F, _P, _P, _P, _P, _SZ, _I64, _INT,
                                       _P], _INT),
    "liger_linear_ce_two_pass_fwd_bwd_async": ([_P, _P, _P, _I64, _I64, _I64, _I64, _INT, _F, _P, _P, _P, _P, _SZ,
                                                _I64, _INT, _P], _INT),
}


class LigerError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def header_functions() -> list:
    """Names of the functions include/liger.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(liger_[a-z_0-9]+)\s*\(", text, re.M)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libliger.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                                   "(python -m transformer_rmsnorm_fwd_gb300.build)")
            lib = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def lib() -> ctypes.CDLL:
    return load()


def _check(rc: int):
    if rc != 0:
        raise LigerError(rc, load().liger_last_error().decode())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return LIGER_F32
    if t.dtype == torch.bfloat16:
        return LIGER_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dense(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ------------------------------------------------------------- device status
def liger_device_status():
    """Waits for the current stream and raises LigerError (LIGER_ERR_CUDA) if a
    bounded wait expired in a kernel of the RMSNorm, RoPE, FusedLinearSwiGLU or
    fused RMSNorm + QKV + RoPE entry points since the last check (the words are
    cleared)."""
    _check(load().liger_device_status(_stream()))


def liger_device_status_mark(which: int):
    """Marks family `which` (0 RMSNorm, 1 FusedLinearSwiGLU, 2 fused QKV, 3 RoPE)
    as an expired wait would, on the current stream (a test hook; nothing expires)."""
    _check(load().liger_device_status_mark(int(which), _stream()))


# ------------------------------------------------------------------ RMSNorm
def liger_rmsnorm_fwd(x, w, y, rstd=None, eps: float = 1e-6):
    _dense(x, w, y, rstd)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    _check(load().liger_rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), rows, cols, eps, _dtype_code(x),
                                    _stream()))
    return y, rstd


def liger_rmsnorm_bwd_workspace(rows: int, cols: int) -> int:
    return int(load().liger_rmsnorm_bwd_workspace(rows, cols))


def liger_rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws):
    _dense(dy, x, w, rstd, dx, dw, ws)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().liger_rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw), _ptr(ws), nbytes,
                                    rows, cols, _dtype_code(x), _stream()))
    return dx, dw


def liger_rmsnorm_bwd_noalloc(dy, x, w, rstd, dx, dw):
    """RMSNorm backward with no workspace argument: the library keeps the
    scratch in its own fixed device array (see liger.h for who needs this and
    the limits: calls that overlap on the GPU share that array)."""
    _dense(dy, x, w, rstd, dx, dw)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    _check(load().liger_rmsnorm_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw), rows, cols,
                                            _dtype_code(x), _stream()))
    return dx, dw


# --------------------------------------------------------------------- RoPE
def _rope(fn, q, k, pos, theta):
    _dense(q, k, pos)
    B, S, Hq, D = q.shape
    Hk = k.shape[2] if k is not None else 0
    if k is not None and (k.shape[0] != B or k.shape[1] != S or k.shape[3] != D):
        raise ValueError("q and k must agree in batch, seq and head_dim")
    _check(fn(_ptr(q), _ptr(k), _ptr(pos), B, S, Hq, Hk, D, float(theta), _dtype_code(q), _stream()))
    return q, k


def liger_rope_fwd(q, k, pos=None, theta: float = 1e4):
    return _rope(load().liger_rope_fwd, q, k, pos, theta)


def liger_rope_bwd(dq, dk, pos=None, theta: float = 1e4):
    return _rope(load().liger_rope_bwd, dq, dk, pos, theta)


def _rope_ex(fn, q, k, q_token_stride, k_token_stride, n_q_heads, n_k_heads, head_dim, batch, seq, pos, theta,
             pairing, cos_tab, sin_tab):
    for t in (pos, cos_tab, sin_tab):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("pos and tables must be contiguous CUDA tensors")
    n_tab = cos_tab.shape[0] if cos_tab is not None else 0
    dt = _dtype_code(q if q is not None else k)
    _check(fn(_ptr(q), _ptr(k), _ptr(pos), batch, seq, n_q_heads, n_k_heads, head_dim, q_token_stride,
              k_token_stride, 1 if pairing == "interleaved" else 0, _ptr(cos_tab), _ptr(sin_tab), n_tab,
              float(theta), dt, _stream()))


def liger_rope_fwd_ex(q, k, q_token_stride, k_token_stride, n_q_heads, n_k_heads, head_dim, batch, seq, pos=None,
                      theta=1e4, pairing="half", cos_tab=None, sin_tab=None):
    """RoPE variants in place on (possibly strided) q / k views: see liger.h.
    q and k are torch tensors whose data_ptr() is the first element of the view."""
    _rope_ex(load().liger_rope_fwd_ex, q, k, q_token_stride, k_token_stride, n_q_heads, n_k_heads, head_dim, batch,
             seq, pos, theta, pairing, cos_tab, sin_tab)


def liger_rope_bwd_ex(dq, dk, q_token_stride, k_token_stride, n_q_heads, n_k_heads, head_dim, batch, seq, pos=None,
                      theta=1e4, pairing="half", cos_tab=None, sin_tab=None):
    _rope_ex(load().liger_rope_bwd_ex, dq, dk, q_token_stride, k_token_stride, n_q_heads, n_k_heads, head_dim, batch,
             seq, pos, theta, pairing, cos_tab, sin_tab)


# ------------------------------------------------------------------- SwiGLU
def liger_swiglu_fwd(gate, up, y):
    _dense(gate, up, y)
    _check(load().liger_swiglu_fwd(_ptr(gate), _ptr(up), _ptr(y), gate.numel(), _dtype_code(gate), _stream()))
    return y


def liger_swiglu_bwd(dy, gate, up, dgate, dup):
    _dense(dy, gate, up, dgate, dup)
    _check(load().liger_swiglu_bwd(_ptr(dy), _ptr(gate), _ptr(up), _ptr(dgate), _ptr(dup), gate.numel(),
                                   _dtype_code(gate), _stream()))
    return dgate, dup


# -------------------------------------------------------- FusedLinearSwiGLU
def liger_fused_linear_swiglu_fwd(X, Wg, Wu, out):
    _dense(X, Wg, Wu, out)
    T, H = X.shape
    I = Wg.shape[0]
    _check(load().liger_fused_linear_swiglu_fwd(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(out), T, H, I, _dtype_code(X),
                                                _stream()))
    return out


def liger_fused_linear_swiglu_workspace(T: int, I: int) -> int:
    return int(load().liger_fused_linear_swiglu_workspace(T, I))


def liger_fused_linear_swiglu_bwd(X, Wg, Wu, dH, dX, dWg, dWu, ws):
    _dense(X, Wg, Wu, dH, dX, dWg, dWu, ws)
    T, H = X.shape
    I = Wg.shape[0]
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().liger_fused_linear_swiglu_bwd(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(dH), _ptr(dX), _ptr(dWg),
                                                _ptr(dWu), _ptr(ws), nbytes, T, H, I, _dtype_code(X), _stream()))
    return dX, dWg, dWu


# ------------------------------------------------ fused RMSNorm + QKV + RoPE
def liger_rmsnorm_qkv_rope_workspace(tokens: int, hidden: int, n_q_heads: int, n_k_heads: int, head_dim: int) -> int:
    return int(load().liger_rmsnorm_qkv_rope_workspace(tokens, hidden, n_q_heads, n_k_heads, head_dim))


def liger_rmsnorm_qkv_rope_fwd(x, w_norm, Wq, Wk, Wv, q, k, v, ws, batch, seq, n_q_heads, n_k_heads, head_dim,
                               bq=None, bk=None, bv=None, pos=None, cos_tab=None, sin_tab=None, rstd=None,
                               eps=1e-6, theta=1e4, folded=False):
    """Fused RMSNorm + QKV projection + RoPE forward (see liger.h): x [B*S, H];
    q [B,S,Hq,D], k and v [B,S,Hk,D] written; folded=True reuses the folded
    weights already in ws."""
    _dense(x, w_norm, Wq, Wk, Wv, bq, bk, bv, pos, cos_tab, sin_tab, q, k, v, rstd, ws)
    H = x.shape[-1]
    n_tab = cos_tab.shape[0] if cos_tab is not None else 0
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().liger_rmsnorm_qkv_rope_fwd(_ptr(x), _ptr(w_norm), _ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(bq), _ptr(bk),
                                             _ptr(bv), _ptr(pos), _ptr(cos_tab), _ptr(sin_tab), n_tab, _ptr(q),
                                             _ptr(k), _ptr(v), _ptr(rstd), _ptr(ws), nbytes, batch, seq, H,
                                             n_q_heads, n_k_heads, head_dim, float(eps), float(theta),
                                             1 if folded else 0, _dtype_code(x), _stream()))
    return q, k, v


def liger_fused_linear_swiglu_fwd_save(X, Wg, Wu, out, g, u):
    """FusedLinearSwiGLU forward that also writes g = X Wg^T and u = X Wu^T."""
    _dense(X, Wg, Wu, out, g, u)
    T, H = X.shape
    I = Wg.shape[0]
    _check(load().liger_fused_linear_swiglu_fwd_save(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(out), _ptr(g), _ptr(u), T, H, I,
                                                     _dtype_code(X), _stream()))
    return out, g, u


def liger_fused_linear_swiglu_bwd_saved(X, Wg, Wu, dH, g, u, dX, dWg, dWu, ws):
    """FusedLinearSwiGLU backward from the g, u the saving forward kept."""
    _dense(X, Wg, Wu, dH, g, u, dX, dWg, dWu, ws)
    T, H = X.shape
    I = Wg.shape[0]
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().liger_fused_linear_swiglu_bwd_saved(_ptr(X), _ptr(Wg), _ptr(Wu), _ptr(dH), _ptr(g), _ptr(u), _ptr(dX),
                                                      _ptr(dWg), _ptr(dWu), _ptr(ws), nbytes, T, H, I, _dtype_code(X),
                                                      _stream()))
    return dX, dWg, dWu


# ---------------------------------------------------------------- linear CE
def liger_linear_ce_workspace(T: int, H: int, V: int, chunk: int = 0, dtype: int = LIGER_BF16) -> int:
    return int(load().liger_linear_ce_workspace(T, H, V, chunk, dtype))


def liger_linear_ce_fwd_bwd(X, W, labels, loss, dX, dW, ws, ignore_index: int = -100, reduction: str = "mean",
                            grad_scale: float = 1.0, chunk: int = 0, wait: bool = True):
    """Fused linear cross-entropy (see liger.h); wait=False calls the _async form
    (no host wait: capturable in a CUDA graph; a bad label makes the loss NaN)."""
    _dense(X, W, labels, loss, dX, dW, ws)
    T, H = X.shape
    V = W.shape[0]
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    fn = load().liger_linear_ce_fwd_bwd if wait else load().liger_linear_ce_fwd_bwd_async
    _check(fn(_ptr(X), _ptr(W), _ptr(labels), T, H, V, int(ignore_index), 0 if reduction == "mean" else 1,
              float(grad_scale), _ptr(loss), _ptr(dX), _ptr(dW), _ptr(ws), nbytes, int(chunk), _dtype_code(X),
              _stream()))
    return loss, dX, dW


def liger_linear_ce_two_pass_workspace(T: int, H: int, V: int, vchunk: int = 0) -> int:
    return int(load().liger_linear_ce_two_pass_workspace(T, H, V, vchunk))


def liger_linear_ce_two_pass_fwd_bwd(X, W, labels, loss, dX, dW, ws, ignore_index: int = -100,
                                     reduction: str = "mean", grad_scale: float = 1.0, vchunk: int = 0,
                                     wait: bool = True):
    """Two-pass, vocabulary-chunked fused linear cross-entropy (see liger.h);
    wait=False calls the _async form."""
    _dense(X, W, labels, loss, dX, dW, ws)
    T, H = X.shape
    V = W.shape[0]
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    fn = load().liger_linear_ce_two_pass_fwd_bwd if wait else load().liger_linear_ce_two_pass_fwd_bwd_async
    _check(fn(_ptr(X), _ptr(W), _ptr(labels), T, H, V, int(ignore_index), 0 if reduction == "mean" else 1,
              float(grad_scale), _ptr(loss), _ptr(dX), _ptr(dW), _ptr(ws), nbytes, int(vchunk), _dtype_code(X),
              _stream()))
    return loss, dX, dW
