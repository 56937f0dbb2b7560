"""Python binding of the split-KV decode attention C ABI (include/decode_attn_splitkv.h).

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libdecode_attn_splitkv.so``. Tensors are PyTorch CUDA tensors
(PyTorch supplies device memory and the stream); they are passed to the
library as raw pointers. There is no CPU fallback: if the library is missing,
importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import math
import os

from .build import LIB, build

DA_OK, DA_ERR_INVALID_ARG, DA_ERR_UNSUPPORTED, DA_ERR_ALIGNMENT = 0, 1, 2, 3
DA_ERR_WORKSPACE_TOO_SMALL, DA_ERR_CUDA, DA_ERR_SCRATCH_LIMIT, DA_ERR_DEVICE_TIMEOUT = 4, 5, 6, 7
DA_F16, DA_BF16 = 0, 1
DA_LAYOUT_VARLEN, DA_LAYOUT_BHSD = 0, 1
DA_LAYOUT_VARLEN_THD = DA_LAYOUT_VARLEN
DA_DEVERR_SEQLENS, DA_DEVERR_TIMEOUT = 0x1, 0x2
DA_MAX_SPLITS = 1024
DA_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
DA_MAX_VARSPLIT_BATCH = 1024
DA_MAX_QUERY_TOKENS = 16

EXPORTED = [
    "decode_attn_splitkv_workspace_size", "decode_attn_splitkv_lse_offset",
    "decode_attn_splitkv_opart_offset", "decode_attn_splitkv_workspace_init",
    "decode_attn_splitkv_num_splits", "decode_attn_splitkv_split_range", "decode_attn_splitkv",
    "decode_attn_splitkv_partial", "decode_attn_splitkv_combine", "decode_attn_splitkv_get_error",
    "decode_attn_splitkv_selftest_timeout", "decode_attn_splitkv_status_string",
    "decode_attn_splitkv_noalloc", "decode_attn_splitkv_varsplit",
    "decode_attn_splitkv_varsplit_plan", "decode_attn_splitkv_multiquery",
    "decode_attn_splitkv_model_us", "decode_attn_splitkv_model_best_splits",
    "decode_attn_splitkv_partial_cuda_core", "decode_attn_splitkv_multiquery_tmem",
    "decode_attn_splitkv_noalloc_get_error", "decode_attn_splitkv_multiquery_varsplit",
    "decode_attn_splitkv_model_varsplit_us",
]

_lib = None


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


def load(path: str = LIB):
    """Load the compiled library (build() first). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                        ctypes.c_float)
    lib.decode_attn_splitkv_workspace_size.argtypes = [I, I, I, I]
    lib.decode_attn_splitkv_workspace_size.restype = SZ
    lib.decode_attn_splitkv_lse_offset.argtypes = []
    lib.decode_attn_splitkv_lse_offset.restype = SZ
    lib.decode_attn_splitkv_opart_offset.argtypes = [I, I, I]
    lib.decode_attn_splitkv_opart_offset.restype = SZ
    lib.decode_attn_splitkv_workspace_init.argtypes = [P, SZ, P]
    lib.decode_attn_splitkv_workspace_init.restype = I
    lib.decode_attn_splitkv_num_splits.argtypes = [I, I, I, I, I, I, I]
    lib.decode_attn_splitkv_num_splits.restype = I
    lib.decode_attn_splitkv_split_range.argtypes = [I64, I, I, ctypes.POINTER(I64),
                                                    ctypes.POINTER(I64)]
    lib.decode_attn_splitkv_split_range.restype = None
    lib.decode_attn_splitkv.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, SZ, P]
    lib.decode_attn_splitkv.restype = I
    lib.decode_attn_splitkv_partial.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, I, P, SZ, P]
    lib.decode_attn_splitkv_partial.restype = I
    lib.decode_attn_splitkv_partial_cuda_core.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, I, P, SZ, P]
    lib.decode_attn_splitkv_partial_cuda_core.restype = I
    lib.decode_attn_splitkv_combine.argtypes = [I, I, I, I, I, P, P, SZ, P]
    lib.decode_attn_splitkv_combine.restype = I
    lib.decode_attn_splitkv_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.decode_attn_splitkv_get_error.restype = I
    lib.decode_attn_splitkv_selftest_timeout.argtypes = [P, SZ, ctypes.c_uint, P]
    lib.decode_attn_splitkv_selftest_timeout.restype = I
    lib.decode_attn_splitkv_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, I, P, P]
    lib.decode_attn_splitkv_noalloc.restype = I
    lib.decode_attn_splitkv_noalloc_get_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.decode_attn_splitkv_noalloc_get_error.restype = I
    lib.decode_attn_splitkv_varsplit.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P, SZ, P]
    lib.decode_attn_splitkv_varsplit.restype = I
    lib.decode_attn_splitkv_varsplit_plan.argtypes = [I, I, I, I, I64, I, I, ctypes.POINTER(I),
                                                      ctypes.POINTER(I)]
    lib.decode_attn_splitkv_varsplit_plan.restype = I
    lib.decode_attn_splitkv_multiquery.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P,
                                                   SZ, P]
    lib.decode_attn_splitkv_multiquery.restype = I
    lib.decode_attn_splitkv_multiquery_varsplit.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P,
                                                            P, SZ, P]
    lib.decode_attn_splitkv_multiquery_varsplit.restype = I
    lib.decode_attn_splitkv_multiquery_tmem.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P,
                                                        SZ, P]
    lib.decode_attn_splitkv_multiquery_tmem.restype = I
    lib.decode_attn_splitkv_model_us.argtypes = [P, I, I, I, I, I, I, I, P]
    lib.decode_attn_splitkv_model_us.restype = ctypes.c_double
    lib.decode_attn_splitkv_model_varsplit_us.argtypes = [P, I, I, I, I, I, I, I, I, P]
    lib.decode_attn_splitkv_model_varsplit_us.restype = ctypes.c_double
    lib.decode_attn_splitkv_model_best_splits.argtypes = [P, I, I, I, I, I, I,
                                                          ctypes.POINTER(ctypes.c_double)]
    lib.decode_attn_splitkv_model_best_splits.restype = I
    lib.decode_attn_splitkv_status_string.argtypes = [I]
    lib.decode_attn_splitkv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != DA_OK:
        raise DecodeAttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return DA_F16
    if t.dtype == torch.bfloat16:
        return DA_BF16
    raise TypeError(f"q/k/v must be float16 or bfloat16, not {t.dtype}")


# ---------------------------------------------------------------- host helpers
def status_string(status: int) -> str:
    return load().decode_attn_splitkv_status_string(status).decode()


def workspace_size(B: int, Hq: int, D: int, num_splits: int) -> int:
    return load().decode_attn_splitkv_workspace_size(B, Hq, D, num_splits)


def num_splits(B: int, Hq: int, Hkv: int, D: int, min_kv: int, max_kv: int, sm_count: int = 0) -> int:
    return load().decode_attn_splitkv_num_splits(B, Hq, Hkv, D, min_kv, max_kv, sm_count)


def split_range(L: int, S: int, s: int) -> tuple:
    a, b = ctypes.c_int64(), ctypes.c_int64()
    load().decode_attn_splitkv_split_range(L, S, s, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def model_us(lens, Hq: int, Hkv: int, D: int, num_splits: int, sm_count: int, T_q: int = 1,
             params=None) -> float:
    """Predicted µs of one call (the GB300 time model; params: 8 values as in the C header,
    None = the built-in calibration)."""
    import numpy as np
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    pa = None if params is None else np.ascontiguousarray(params, dtype=np.float64)
    if pa is not None and pa.size != 8:
        raise ValueError("model_us takes 8 parameters")
    return load().decode_attn_splitkv_model_us(ln.ctypes.data, ln.size, Hq, Hkv, D, T_q, num_splits,
                                               sm_count, None if pa is None else pa.ctypes.data)


def model_varsplit_us(lens, Hq: int, Hkv: int, D: int, split_len: int, max_splits: int, sm_count: int,
                      T_q: int = 1, params=None) -> float:
    """Predicted µs of one call with per-sequence split counts (the same model)."""
    import numpy as np
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    pa = None if params is None else np.ascontiguousarray(params, dtype=np.float64)
    if pa is not None and pa.size != 8:
        raise ValueError("model_varsplit_us takes 8 parameters")
    return load().decode_attn_splitkv_model_varsplit_us(ln.ctypes.data, ln.size, Hq, Hkv, D, T_q, split_len,
                                                        max_splits, sm_count,
                                                        None if pa is None else pa.ctypes.data)


def model_best_splits(lens, Hq: int, Hkv: int, D: int, sm_count: int, T_q: int = 1) -> tuple:
    """(split count, predicted µs) minimising the GB300 time model."""
    import numpy as np
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    t = ctypes.c_double()
    S = load().decode_attn_splitkv_model_best_splits(ln.ctypes.data, ln.size, Hq, Hkv, D, T_q, sm_count,
                                                     ctypes.byref(t))
    return S, t.value


def alloc_workspace(B: int, Hq: int, D: int, num_splits_: int, device="cuda", stream=None):
    """Allocate (through PyTorch) and initialise a workspace for these sizes."""
    import torch
    nbytes = workspace_size(B, Hq, D, num_splits_)
    if nbytes == 0:
        raise ValueError("workspace_size rejected the sizes")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check(load().decode_attn_splitkv_workspace_init(_ptr(ws), nbytes, _stream(stream)),
           "decode_attn_splitkv_workspace_init")
    return ws


def workspace_views(ws, B: int, Hq: int, D: int, num_splits_: int):
    """(lse_part[B,Hq,S], o_part[B,Hq,S,D]) float32 views into a workspace tensor."""
    import torch
    lib = load()
    lo = lib.decode_attn_splitkv_lse_offset()
    oo = lib.decode_attn_splitkv_opart_offset(B, Hq, num_splits_)
    n = B * Hq * num_splits_
    lse = ws[lo: lo + 4 * n].view(torch.float32).view(B, Hq, num_splits_)
    opart = ws[oo: oo + 4 * n * D].view(torch.float32).view(B, Hq, num_splits_, D)
    return lse, opart


# ---------------------------------------------------------------- device calls
def _shape_args(q, k, cu_seqlens_k, layout):
    B, Hq, D = q.shape
    if layout == DA_LAYOUT_VARLEN:
        kv_rows, Hkv = k.shape[0], k.shape[1]
    else:
        Hkv, kv_rows = k.shape[1], k.shape[2]
    return B, Hq, Hkv, D, kv_rows


def decode_attn_splitkv(q, k, v, cu_seqlens_k, out, workspace, *, num_splits: int,
                        scale: float | None = None, layout: int = DA_LAYOUT_VARLEN, stream=None):
    """out[B,Hq,D] = split-KV decode attention of q over (k, v); see the C header."""
    B, Hq, Hkv, D, kv_rows = _shape_args(q, k, cu_seqlens_k, layout)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, num_splits, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "decode_attn_splitkv")
    return out


def varsplit_plan(B: int, Hq: int, Hkv: int, D: int, total_kv: int, max_kv: int,
                  sm_count: int = 0) -> tuple:
    """(split_len, max_splits) for decode_attn_splitkv_varsplit."""
    a, b = ctypes.c_int(), ctypes.c_int()
    rc = load().decode_attn_splitkv_varsplit_plan(B, Hq, Hkv, D, total_kv, max_kv, sm_count,
                                                  ctypes.byref(a), ctypes.byref(b))
    if rc != 0:
        raise ValueError("decode_attn_splitkv_varsplit_plan rejected its arguments")
    return a.value, b.value


def decode_attn_splitkv_varsplit(q, k, v, cu_seqlens_k, out, workspace, *, split_len: int,
                                 max_splits: int, scale: float | None = None,
                                 layout: int = DA_LAYOUT_VARLEN, stream=None):
    """Per-sequence split counts S_b = min(max_splits, ceil(L_b / split_len)); see the C header."""
    B, Hq, Hkv, D, kv_rows = _shape_args(q, k, cu_seqlens_k, layout)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv_varsplit(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, split_len, max_splits, _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(st, "decode_attn_splitkv_varsplit")
    return out


def _multiquery(name, q, k, v, cu_seqlens_k, out, workspace, num_splits, scale, layout, stream):
    B, T, Hq, D = q.shape
    if layout == DA_LAYOUT_VARLEN:
        kv_rows, Hkv = k.shape[0], k.shape[1]
    else:
        Hkv, kv_rows = k.shape[1], k.shape[2]
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = getattr(load(), name)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, T, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, num_splits, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, name)
    return out


def decode_attn_splitkv_multiquery(q, k, v, cu_seqlens_k, out, workspace, *, num_splits: int,
                                   scale: float | None = None, layout: int = DA_LAYOUT_VARLEN,
                                   stream=None):
    """Several query tokens per sequence: q and out are [B, T_q, Hq, D]; see the C header."""
    return _multiquery("decode_attn_splitkv_multiquery", q, k, v, cu_seqlens_k, out, workspace, num_splits,
                       scale, layout, stream)


def decode_attn_splitkv_multiquery_varsplit(q, k, v, cu_seqlens_k, out, workspace, *, split_len: int,
                                            max_splits: int, scale: float | None = None,
                                            layout: int = DA_LAYOUT_VARLEN, stream=None):
    """Several query tokens per sequence with per-sequence split counts: q and out are
    [B, T_q, Hq, D]; see the C header."""
    B, T, Hq, D = q.shape
    if layout == DA_LAYOUT_VARLEN:
        kv_rows, Hkv = k.shape[0], k.shape[1]
    else:
        Hkv, kv_rows = k.shape[1], k.shape[2]
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv_multiquery_varsplit(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, T, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, split_len, max_splits, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "decode_attn_splitkv_multiquery_varsplit")
    return out


def decode_attn_splitkv_multiquery_tmem(q, k, v, cu_seqlens_k, out, workspace, *, num_splits: int,
                                        scale: float | None = None, layout: int = DA_LAYOUT_VARLEN,
                                        stream=None):
    """The tcgen05 / tensor-memory comparison arm of decode_attn_splitkv_multiquery (G * T_q > 8,
    G <= 32); see the C header."""
    return _multiquery("decode_attn_splitkv_multiquery_tmem", q, k, v, cu_seqlens_k, out, workspace,
                       num_splits, scale, layout, stream)


def decode_attn_splitkv_partial(q, k, v, cu_seqlens_k, workspace, *, num_splits: int,
                                scale: float | None = None, layout: int = DA_LAYOUT_VARLEN,
                                stream=None):
    B, Hq, Hkv, D, kv_rows = _shape_args(q, k, cu_seqlens_k, layout)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv_partial(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, num_splits, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "decode_attn_splitkv_partial")


def decode_attn_splitkv_partial_cuda_core(q, k, v, cu_seqlens_k, workspace, *, num_splits: int,
                                          scale: float | None = None, layout: int = DA_LAYOUT_VARLEN,
                                          stream=None):
    """The split step with CUDA-core FMA products (comparison arm); see the C header."""
    B, Hq, Hkv, D, kv_rows = _shape_args(q, k, cu_seqlens_k, layout)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv_partial_cuda_core(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, num_splits, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "decode_attn_splitkv_partial_cuda_core")


def decode_attn_splitkv_combine(out, workspace, *, num_splits: int, stream=None):
    B, Hq, D = out.shape
    st = load().decode_attn_splitkv_combine(B, Hq, D, num_splits, _dtype_code(out), _ptr(out),
                                            _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "decode_attn_splitkv_combine")
    return out


def decode_attn_splitkv_get_error(workspace, stream=None) -> int:
    """Read and clear the workspace's device error word: the DA_DEVERR_* bits (0 if none).

    A time-out (the C call's DA_ERR_DEVICE_TIMEOUT) is reported through the bits too,
    not raised, so that the caller can tell it from a failed read."""
    bits = ctypes.c_uint32(0)
    st = load().decode_attn_splitkv_get_error(_ptr(workspace), ctypes.byref(bits), _stream(stream))
    if st != DA_ERR_DEVICE_TIMEOUT:
        _check(st, "decode_attn_splitkv_get_error")
    return bits.value


def decode_attn_splitkv_noalloc_get_error(stream=None) -> int:
    """decode_attn_splitkv_get_error for decode_attn_splitkv_noalloc's built-in scratch array."""
    bits = ctypes.c_uint32(0)
    st = load().decode_attn_splitkv_noalloc_get_error(ctypes.byref(bits), _stream(stream))
    if st != DA_ERR_DEVICE_TIMEOUT:
        _check(st, "decode_attn_splitkv_noalloc_get_error")
    return bits.value


def decode_attn_splitkv_selftest_timeout(workspace, timeout_us: int, stream=None) -> None:
    _check(load().decode_attn_splitkv_selftest_timeout(_ptr(workspace), workspace.numel(),
                                                       timeout_us, _stream(stream)),
           "decode_attn_splitkv_selftest_timeout")


def decode_attn_splitkv_noalloc(q, k, v, cu_seqlens_k, out, *, num_splits: int,
                                scale: float | None = None, layout: int = DA_LAYOUT_VARLEN,
                                stream=None):
    """decode_attn_splitkv with the library's built-in scratch array instead of a workspace.

    For callers that may not allocate device memory (a plugin interface that
    owns all allocation, or a path where cudaMalloc's device-wide
    synchronisation is not acceptable). Problems needing more than
    DA_NOALLOC_SCRATCH_BYTES of scratch raise DecodeAttnError
    (DA_ERR_SCRATCH_LIMIT). Calls share the array: do not let them overlap.
    """
    B, Hq, Hkv, D, kv_rows = _shape_args(q, k, cu_seqlens_k, layout)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    st = load().decode_attn_splitkv_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), B, Hq, Hkv, D, kv_rows, _dtype_code(q),
        layout, sc, num_splits, _ptr(out), _stream(stream))
    _check(st, "decode_attn_splitkv_noalloc")
    return out
