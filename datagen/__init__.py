"""Seeded synthetic inputs, shared by the fp64 oracle and the CUDA path.

This package holds no operator arithmetic: only the counter-based random
draws of ``gen.c`` (SplitMix64 streams keyed by tensor name, Box-Muller
normals, Lemire labels, Fisher-Yates ignore rows) and the workload recipes
that name each tensor, its shape and its distribution.

``build()`` compiles ``gen.c`` with gcc into ``libdatagen.so`` next to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libdatagen.so")
_lib = None
_lock = threading.Lock()

F64, F32, BF16 = 0, 1, 2
_DTYPE_CODE = {"f64": F64, "f32": F32, "bf16": BF16}


def build(force: bool = False) -> str:
    """Compile gen.c into libdatagen.so (gcc, -O2, pthreads)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.gen_normal.argtypes = [ctypes.c_uint64, ctypes.c_char_p, ctypes.c_double, ctypes.c_double,
                                       ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int]
            lib.gen_normal.restype = ctypes.c_int
            lib.gen_labels.argtypes = [ctypes.c_uint64, ctypes.c_char_p, ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
            lib.gen_labels.restype = ctypes.c_int
            lib.gen_positions.argtypes = [ctypes.c_uint64, ctypes.c_char_p, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int64]
            lib.gen_positions.restype = ctypes.c_int
            lib.gen_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.gen_draw.restype = ctypes.c_uint64
            lib.gen_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_char_p]
            lib.gen_stream_key.restype = ctypes.c_uint64
            lib.gen_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.gen_f32_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal(seed: int, name: str, shape, dtype: str = "f32", mean: float = 0.0, std: float = 1.0,
           out: np.ndarray | None = None) -> np.ndarray:
    """mean + std * N(0,1), stream (seed, name).  bf16 comes back as uint16 bits."""
    lib = _load()
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = int(np.prod(shape)) if shape else 1
    npdt = {"f64": np.float64, "f32": np.float32, "bf16": np.uint16}[dtype]
    if out is None:
        out = np.empty(shape, dtype=npdt)
    assert out.dtype == npdt and out.size == n and out.flags.c_contiguous
    rc = lib.gen_normal(ctypes.c_uint64(seed & (2**64 - 1)), name.encode(), float(mean), float(std),
                        _DTYPE_CODE[dtype], out.ctypes.data, n, _threads())
    if rc != 0:
        raise ValueError("gen_normal rejected its arguments")
    return out


def labels(seed: int, name: str, T: int, V: int, ignore_frac: float, ignore_index: int = -100) -> np.ndarray:
    """Uniform labels in [0, V) with exactly round(ignore_frac*T) rows set to ignore_index."""
    lib = _load()
    out = np.empty((int(T),), dtype=np.int64)
    n_ignore = int(round(ignore_frac * T))
    rc = lib.gen_labels(ctypes.c_uint64(seed & (2**64 - 1)), name.encode(), out.ctypes.data, int(T), int(V),
                        n_ignore, int(ignore_index))
    if rc != 0:
        raise ValueError("gen_labels rejected its arguments")
    return out


def positions(seed: int, name: str, shape, max_pos: int) -> np.ndarray:
    """int32 positions uniform in [0, max_pos)."""
    lib = _load()
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.int32)
    rc = lib.gen_positions(ctypes.c_uint64(seed & (2**64 - 1)), name.encode(), out.ctypes.data, out.size,
                           int(max_pos))
    if rc != 0:
        raise ValueError("gen_positions rejected its arguments")
    return out


def draw(seed: int, name: str, i: int) -> int:
    """Raw 64-bit draw i of stream (seed, name) (for checking the generator)."""
    lib = _load()
    key = lib.gen_stream_key(ctypes.c_uint64(seed & (2**64 - 1)), name.encode())
    return int(lib.gen_draw(key, int(i)))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even), returning uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7F800000) == 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = (u[nan] >> 16).astype(np.uint16) | np.where((u[nan] & 0x7FFFFF) != 0, 0x40, 0).astype(np.uint16)
    return r


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored values (f32, f64 or bf16 bits) exactly to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


from . import workloads  # noqa: E402,F401
