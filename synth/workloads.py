"""Named decode-attention workloads and their seeded inputs.

Every workload is one decode step: one query token per sequence, ``Hq``
query heads sharing ``Hkv`` KV heads, head size ``D``, and a KV cache whose
per-sequence lengths are given by ``cu_seqlens_k`` (prefix sums of the
lengths). Two cache layouts exist:

* ``varlen``: K and V are ``[total_kv, Hkv, D]``; sequence b owns rows
  ``cu[b] .. cu[b+1]-1``.
* ``bhsd``: K and V are ``[B, Hkv, kv_rows, D]``; sequence b owns positions
  ``0 .. cu[b+1]-cu[b]-1`` of its own slab (``kv_rows`` is the capacity).

Values are N(0, 1) draws rounded to binary16 or bfloat16 (``synth.normal_bits``),
from stream 1 (Q), 2 (K), 3 (V); varlen lengths come from stream 4. The shapes
follow the workloads the split-KV decoding pages discuss: the Triton self-test
shape, the TileLang default shape (Qwen2.5-7B heads), the flash-decoding blog's
CodeLlama-34B microbenchmark sweep and the Llama-3.1-8B long-context table.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import normal_bits, uniform_int

LAYOUT_VARLEN, LAYOUT_BHSD = 0, 1
DTYPE_F16, DTYPE_BF16 = 0, 1


@dataclass
class Problem:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    lens: list
    dtype: str          # "f16" or "bf16"
    layout: int         # LAYOUT_VARLEN or LAYOUT_BHSD
    scale: float
    num_splits: int | None   # None: use the split-count picker
    seed: int = 0
    kv_rows: int = 0
    tq: int = 1              # query tokens per sequence; q is [B, tq, Hq, D] when tq > 1
    q: np.ndarray | None = field(default=None, repr=False)
    k: np.ndarray | None = field(default=None, repr=False)
    v: np.ndarray | None = field(default=None, repr=False)
    cu: np.ndarray | None = field(default=None, repr=False)

    @property
    def dtype_code(self) -> int:
        return DTYPE_F16 if self.dtype == "f16" else DTYPE_BF16

    @property
    def total_kv(self) -> int:
        return int(sum(self.lens))

    @property
    def kv_bytes(self) -> int:
        """K plus V bytes the method must read: 2 * sum(L_b) * Hkv * D * 2."""
        return 2 * self.total_kv * self.Hkv * self.D * 2

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


def cu_from_lens(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64)).astype(np.int32)
    return cu


def materialize(p: Problem, q_mean: float = 0.0, q_std: float = 1.0,
                k_mean: float = 0.0, k_std: float = 1.0,
                v_mean: float = 0.0, v_std: float = 1.0) -> Problem:
    """Fill p.q, p.k, p.v (uint16 bit patterns) and p.cu (int32) from the seed."""
    p.cu = cu_from_lens(p.lens)
    if p.layout == LAYOUT_VARLEN:
        p.kv_rows = p.total_kv
        kv_shape = (p.kv_rows, p.Hkv, p.D)
    else:
        if p.kv_rows < max(p.lens, default=0):
            p.kv_rows = max(p.lens, default=0)
        kv_shape = (p.B, p.Hkv, p.kv_rows, p.D)
    nq = p.B * p.tq * p.Hq * p.D
    q_shape = (p.B, p.Hq, p.D) if p.tq == 1 else (p.B, p.tq, p.Hq, p.D)
    nkv = int(np.prod(kv_shape))
    p.q = normal_bits(p.seed, 1, nq, p.dtype, q_mean, q_std).reshape(q_shape)
    p.k = normal_bits(p.seed, 2, nkv, p.dtype, k_mean, k_std).reshape(kv_shape)
    p.v = normal_bits(p.seed, 3, nkv, p.dtype, v_mean, v_std).reshape(kv_shape)
    return p


def custom(name, B, Hq, Hkv, D, lens, dtype="f16", layout=LAYOUT_VARLEN, num_splits=None,
           seed=0, kv_rows=0, scale=None, data=True, tq=1, **dist) -> Problem:
    p = Problem(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, lens=[int(x) for x in lens], dtype=dtype,
                layout=layout, scale=(1.0 / math.sqrt(D)) if scale is None else scale,
                num_splits=num_splits, seed=seed, kv_rows=kv_rows, tq=tq)
    if data:
        materialize(p, **dist)
    return p


def qwen_lengths(B: int, seed: int = 0, lo: int = 512, hi: int = 8192) -> list:
    return [int(x) for x in uniform_int(seed, 4, B, lo, hi)]


# (batch, seqlen) pairs of the CodeLlama-34B-shaped sweep (constant batch*seqlen, plus 128K).
CODELLAMA_SWEEP = [(256, 256), (128, 512), (64, 1024), (32, 2048), (16, 4096), (8, 8192),
                   (4, 16384), (2, 32768), (1, 65536), (1, 131072)]
# (seqlen, batch) pairs of the Llama-3.1-8B long-context table.
LLAMA_SWEEP = [(s, b) for s in (1024, 8192, 32768, 131072) for b in (1, 16)]


def workload(name: str, data: bool = True, seed: int = 0) -> Problem:
    """Build a named workload.

    tiny                 B=2, 4 q / 1 kv heads, D=64, lengths [37, 200], fp16, 4 splits
    mha_bhsd             B=8, 32 q = 32 kv heads, D=128, every length 4096, fp16, bhsd layout
    qwen_varlen          B=64, 28 q / 4 kv heads, D=128, lengths uniform on [512, 8192], fp16
    codellama_B{b}_S{s}  16 q / 2 kv heads, D=128, b sequences of length s, fp16
    llama_S{s}_B{b}      32 q / 8 kv heads, D=128, b sequences of length s, bf16
    llama_skewed         32 q / 8 kv heads, D=128, bf16, one sequence of 131072 and 15 of 512
    """
    if name == "tiny":
        return custom(name, 2, 4, 1, 64, [37, 200], "f16", LAYOUT_VARLEN, 4, seed, data=data)
    if name == "mha_bhsd":
        return custom(name, 8, 32, 32, 128, [4096] * 8, "f16", LAYOUT_BHSD, None, seed,
                      kv_rows=4096, data=data)
    if name == "qwen_varlen":
        return custom(name, 64, 28, 4, 128, qwen_lengths(64, seed), "f16", LAYOUT_VARLEN,
                      None, seed, data=data)
    if name.startswith("codellama_B"):
        b, s = name[len("codellama_B"):].split("_S")
        return custom(name, int(b), 16, 2, 128, [int(s)] * int(b), "f16", LAYOUT_VARLEN,
                      None, seed, data=data)
    if name == "llama_skewed":
        # one long-context sequence in a batch of short ones: the case per-sequence
        # split counts are for (a uniform count is capped by the shortest sequence)
        return custom(name, 16, 32, 8, 128, [131072] + [512] * 15, "bf16", LAYOUT_VARLEN, None,
                      seed, data=data)
    if name.startswith("llama_S"):
        s, b = name[len("llama_S"):].split("_B")
        return custom(name, int(b), 32, 8, 128, [int(s)] * int(b), "bf16", LAYOUT_VARLEN,
                      None, seed, data=data)
    raise KeyError(name)


def all_workload_names() -> list:
    names = ["tiny", "mha_bhsd", "qwen_varlen"]
    names += [f"codellama_B{b}_S{s}" for b, s in CODELLAMA_SWEEP]
    names += [f"llama_S{s}_B{b}" for s, b in LLAMA_SWEEP]
    return names
