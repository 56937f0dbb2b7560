"""Float64 CPU oracle for split-KV decode attention (ctypes binding of oracle.cpp).

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and bench.py's CPU-baseline
leg may import this package; the product path (the CUDA library and its
Python binding) never does. It shares no code with the CUDA path.

Parity unpinned: none of its functions. Each is pinned in tests/test_oracle.py
by closed forms, special cases, a library cross-check and split invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def compile_library(src: str, out: str) -> str:
    """g++ -O2 a float64 oracle source into a shared library (plain host C++)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", tmp, src, "-lpthread"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


_P = ctypes.c_void_p
_I32, _I64, _F64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
_PROBLEM_ARGS = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I64, _I32, _I32, _F64]


def load_library(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double.restype = _F64
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = _F64
    lib.oracle_split_range.argtypes = [_I64, _I64, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]
    lib.oracle_split_range.restype = None
    lib.oracle_attention.argtypes = _PROBLEM_ARGS + [_P, _P, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = _PROBLEM_ARGS + [_P, _P, _I32, _P, _P, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_split_partials.argtypes = _PROBLEM_ARGS + [_I32, _P, _P, ctypes.c_int]
    lib.oracle_split_partials.restype = ctypes.c_int
    lib.oracle_split_partials_var.argtypes = _PROBLEM_ARGS + [_I32, _I32, _P, _P, _P, ctypes.c_int]
    lib.oracle_split_partials_var.restype = ctypes.c_int
    lib.oracle_attention_mq.argtypes = _PROBLEM_ARGS + [_I32, _P, _P, ctypes.c_int]
    lib.oracle_attention_mq.restype = ctypes.c_int
    lib.oracle_attention_rows_mq.argtypes = _PROBLEM_ARGS + [_I32, _P, _P, _P, _I32, _P, _P,
                                                             ctypes.c_int]
    lib.oracle_attention_rows_mq.restype = ctypes.c_int
    lib.oracle_split_partials_mq.argtypes = _PROBLEM_ARGS + [_I32, _I32, _P, _P, ctypes.c_int]
    lib.oracle_split_partials_mq.restype = ctypes.c_int
    lib.oracle_split_partials_var_mq.argtypes = _PROBLEM_ARGS + [_I32, _I32, _I32, _P, _P, _P, ctypes.c_int]
    lib.oracle_split_partials_var_mq.restype = ctypes.c_int
    lib.oracle_merge.argtypes = [_P, _P, _I64, _I32, _I32, _P, _P]
    lib.oracle_merge.restype = ctypes.c_int
    lib.oracle_weights.argtypes = _PROBLEM_ARGS + [_I32, _I32, _P]
    lib.oracle_weights.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _threads(nthreads):
    return nthreads if nthreads else max(1, os.cpu_count() or 1)


class Oracle:
    """Oracle bound to one compiled library (the real one, or a test's planted variant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else _load()

    # ---- encodings -------------------------------------------------------
    def f16_to_double(self, bits: int) -> float:
        return self.lib.oracle_f16_to_double(bits)

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(bits)

    def split_range(self, L: int, S: int, s: int) -> tuple:
        a, b = _I64(), _I64()
        self.lib.oracle_split_range(L, S, s, ctypes.byref(a), ctypes.byref(b))
        return a.value, b.value

    # ---- attention ---------------------------------------------------------
    @staticmethod
    def _args(p):
        q = np.ascontiguousarray(p.q)
        k = np.ascontiguousarray(p.k)
        v = np.ascontiguousarray(p.v)
        cu = np.ascontiguousarray(p.cu, dtype=np.int32)
        keep = (q, k, v, cu)
        args = [q.ctypes.data, k.ctypes.data, v.ctypes.data, cu.ctypes.data, p.B, p.Hq, p.Hkv,
                p.D, p.kv_rows, 0 if p.dtype == "f16" else 1, p.layout, p.scale]
        return keep, args

    def attention(self, p, nthreads: int = 0):
        """Plain definition: (out[B,Hq,D], lse[B,Hq]) in float64."""
        keep, args = self._args(p)
        out = np.empty((p.B, p.Hq, p.D), dtype=np.float64)
        lse = np.empty((p.B, p.Hq), dtype=np.float64)
        rc = self.lib.oracle_attention(*args, out.ctypes.data, lse.ctypes.data, _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_attention: inconsistent problem")
        return out, lse

    def attention_rows(self, p, rows_b, rows_h, nthreads: int = 0):
        """Plain definition on sampled (b, h) pairs: (out[n,D], lse[n])."""
        keep, args = self._args(p)
        rb = np.ascontiguousarray(rows_b, dtype=np.int32)
        rh = np.ascontiguousarray(rows_h, dtype=np.int32)
        n = rb.size
        out = np.empty((n, p.D), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64)
        rc = self.lib.oracle_attention_rows(*args, rb.ctypes.data, rh.ctypes.data, n,
                                            out.ctypes.data, lse.ctypes.data, _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_attention_rows: inconsistent problem")
        return out, lse

    def split_partials(self, p, S: int, nthreads: int = 0):
        """Per-split values: (o_part[B,Hq,S,D], lse_part[B,Hq,S])."""
        keep, args = self._args(p)
        o = np.empty((p.B, p.Hq, S, p.D), dtype=np.float64)
        lse = np.empty((p.B, p.Hq, S), dtype=np.float64)
        rc = self.lib.oracle_split_partials(*args, S, o.ctypes.data, lse.ctypes.data,
                                            _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_split_partials: inconsistent problem")
        return o, lse

    def split_partials_var(self, p, split_len: int, max_splits: int, nthreads: int = 0):
        """Per-sequence split counts: (o_part[B,Hq,max_splits,D], lse_part[B,Hq,max_splits], S_b[B])."""
        keep, args = self._args(p)
        o = np.empty((p.B, p.Hq, max_splits, p.D), dtype=np.float64)
        lse = np.empty((p.B, p.Hq, max_splits), dtype=np.float64)
        sc = np.empty(p.B, dtype=np.int32)
        rc = self.lib.oracle_split_partials_var(*args, split_len, max_splits, o.ctypes.data,
                                                lse.ctypes.data, sc.ctypes.data, _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_split_partials_var: inconsistent problem")
        return o, lse, sc

    # ---- several query tokens per sequence (q, out [B, tq, Hq, D]) ----------
    def attention_mq(self, p, tq: int, nthreads: int = 0):
        """Causal multi-token decode: (out[B,tq,Hq,D], lse[B,tq,Hq])."""
        keep, args = self._args(p)
        out = np.empty((p.B, tq, p.Hq, p.D), dtype=np.float64)
        lse = np.empty((p.B, tq, p.Hq), dtype=np.float64)
        rc = self.lib.oracle_attention_mq(*args, tq, out.ctypes.data, lse.ctypes.data,
                                          _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_attention_mq: inconsistent problem")
        return out, lse

    def attention_rows_mq(self, p, tq: int, rows_b, rows_t, rows_h, nthreads: int = 0):
        keep, args = self._args(p)
        rb = np.ascontiguousarray(rows_b, dtype=np.int32)
        rt = np.ascontiguousarray(rows_t, dtype=np.int32)
        rh = np.ascontiguousarray(rows_h, dtype=np.int32)
        out = np.empty((rb.size, p.D), dtype=np.float64)
        lse = np.empty(rb.size, dtype=np.float64)
        rc = self.lib.oracle_attention_rows_mq(*args, tq, rb.ctypes.data, rt.ctypes.data,
                                               rh.ctypes.data, rb.size, out.ctypes.data,
                                               lse.ctypes.data, _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_attention_rows_mq: inconsistent problem")
        return out, lse

    def split_partials_var_mq(self, p, tq: int, split_len: int, max_splits: int, nthreads: int = 0):
        """Per-sequence split counts with tq tokens: (o_part[B,tq,Hq,max_splits,D],
        lse_part[B,tq,Hq,max_splits], S_b[B])."""
        keep, args = self._args(p)
        o = np.empty((p.B, tq, p.Hq, max_splits, p.D), dtype=np.float64)
        lse = np.empty((p.B, tq, p.Hq, max_splits), dtype=np.float64)
        sc = np.empty(p.B, dtype=np.int32)
        rc = self.lib.oracle_split_partials_var_mq(*args, tq, split_len, max_splits, o.ctypes.data,
                                                   lse.ctypes.data, sc.ctypes.data, _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_split_partials_var_mq: inconsistent problem")
        return o, lse, sc

    def split_partials_mq(self, p, tq: int, S: int, nthreads: int = 0):
        """(o_part[B,tq,Hq,S,D], lse_part[B,tq,Hq,S])."""
        keep, args = self._args(p)
        o = np.empty((p.B, tq, p.Hq, S, p.D), dtype=np.float64)
        lse = np.empty((p.B, tq, p.Hq, S), dtype=np.float64)
        rc = self.lib.oracle_split_partials_mq(*args, tq, S, o.ctypes.data, lse.ctypes.data,
                                               _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_split_partials_mq: inconsistent problem")
        return o, lse

    def merge(self, o_part, lse_part):
        """Exact log-sum-exp combine: (out[..., D], lse[...])."""
        o_part = np.ascontiguousarray(o_part, dtype=np.float64)
        lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
        S, D = o_part.shape[-2], o_part.shape[-1]
        lead = o_part.shape[:-2]
        rows = int(np.prod(lead)) if lead else 1
        out = np.empty(lead + (D,), dtype=np.float64)
        lse = np.empty(lead, dtype=np.float64)
        rc = self.lib.oracle_merge(o_part.ctypes.data, lse_part.ctypes.data, rows, S, D,
                                   out.ctypes.data, lse.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_merge: bad shape")
        return out, lse

    def weights(self, p, b: int, h: int):
        keep, args = self._args(p)
        L = int(p.cu[b + 1] - p.cu[b])
        w = np.empty(max(L, 1), dtype=np.float64)
        rc = self.lib.oracle_weights(*args, b, h, w.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_weights: inconsistent problem")
        return w[:L]


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
