"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds none of the attention arithmetic: it produces the bytes of
Q, K, V (binary16 or bfloat16 bit patterns of N(0, 1) draws) and the KV
lengths, from a counter-based generator implemented in ``synth.c``. Both the
float64 oracle and the CUDA path read the identical bytes it returns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

KIND_F16, KIND_BF16, KIND_F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library with gcc (host code, any CPU)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                    "-lm", "-lpthread"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_int, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal.restype = ctypes.c_int
        lib.synth_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_void_p]
        lib.synth_uniform_int.restype = ctypes.c_int
        lib.synth_double_to_f16.argtypes = [ctypes.c_double]
        lib.synth_double_to_f16.restype = ctypes.c_uint16
        lib.synth_double_to_bf16.argtypes = [ctypes.c_double]
        lib.synth_double_to_bf16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bits(seed: int, stream: int, n: int, dtype: str, mean: float = 0.0,
                std: float = 1.0, first: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """n draws of N(mean, std^2) rounded to ``dtype`` ("f16" or "bf16"), as uint16 bits."""
    kind = {"f16": KIND_F16, "bf16": KIND_BF16}[dtype]
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == n and out.flags.c_contiguous
    rc = _load().synth_normal(seed, stream, first, n, kind, mean, std,
                              out.ctypes.data if n else None, _threads())
    if rc != 0:
        raise ValueError("synth_normal rejected its arguments")
    return out


def normal_f64(seed: int, stream: int, n: int, first: int = 0) -> np.ndarray:
    """n unrounded N(0, 1) draws (the values before the dtype rounding)."""
    out = np.empty(n, dtype=np.float64)
    rc = _load().synth_normal(seed, stream, first, n, KIND_F64, 0.0, 1.0,
                              out.ctypes.data if n else None, _threads())
    if rc != 0:
        raise ValueError("synth_normal rejected its arguments")
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, first: int = 0) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive)."""
    out = np.empty(n, dtype=np.int64)
    rc = _load().synth_uniform_int(seed, stream, first, n, lo, hi,
                                   out.ctypes.data if n else None)
    if rc != 0:
        raise ValueError("synth_uniform_int rejected its arguments")
    return out


def round_f16(x: float) -> int:
    return int(_load().synth_double_to_f16(float(x)))


def round_bf16(x: float) -> int:
    return int(_load().synth_double_to_bf16(float(x)))
