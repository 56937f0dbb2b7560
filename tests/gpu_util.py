"""Helpers for the GPU parity tests: move a synthetic problem to the device, run the
CUDA path through the C ABI, and derive tolerances from the arithmetic."""
import numpy as np
import torch

import split_kv_decode_decoding_gb300 as da
from synth.workloads import LAYOUT_VARLEN

# Parity bounds fixed for this method: final output max |delta| (fp16/bf16 outputs)
# and per-split log-sum-exp max |delta| (fp32).
OUT_TOL = 4e-3
LSE_TOL = 1e-4


def opart_tol(p) -> float:
    """Bound for the fp32 per-split outputs.

    The kernel rounds the softmax weights P to the input dtype before the PV
    tensor-core product (unit roundoff u = 2^-11 for fp16, 2^-8 for bf16, so a
    relative error of at most u/2... u per weight), which moves o_s by at most
    u * max|v|; fp32 accumulation and the exp2 approximation add far less.
    """
    u = 2.0 ** -11 if p.dtype == "f16" else 2.0 ** -8
    return u * max_abs_finite(p.v, p.dtype) + 1e-5


def max_abs_finite(bits, dtype: str) -> float:
    """Largest |x| over the finite binary16/bfloat16 values among `bits` (uint16 patterns),
    without widening the whole array: with the sign bit cleared, the bit patterns of finite
    values order like their magnitudes, and Inf/NaN patterns sit above the largest finite one."""
    if bits.size == 0:
        return 1.0
    inf_bits = 0x7C00 if dtype == "f16" else 0x7F80
    mag = np.bitwise_and(np.asarray(bits, dtype=np.uint16).reshape(-1), 0x7FFF)
    finite = mag[mag < inf_bits]
    if finite.size == 0:
        return 1.0
    top = np.array([finite.max()], dtype=np.uint16)
    return float(_decode(top, dtype)[0])


def _decode(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).to(torch.float64).numpy()


def torch_dtype(p):
    return torch.float16 if p.dtype == "f16" else torch.bfloat16


def to_device(p, device="cuda"):
    dt = torch_dtype(p)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt).to(device)

    return dev(p.q), dev(p.k), dev(p.v), torch.from_numpy(p.cu.astype(np.int32)).to(device)


def run(p, S, device="cuda", stream=None, tensors=None):
    """Run the full call; returns (out, lse_part, o_part, error_bits) as float64 numpy."""
    q, k, v, cu = tensors if tensors is not None else to_device(p, device)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, S, device=device, stream=stream)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch_dtype(p), device=device)
    da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale, layout=p.layout,
                           stream=stream)
    err = da.decode_attn_splitkv_get_error(ws, stream=stream)
    lse, opart = da.workspace_views(ws, p.B, p.Hq, p.D, S)
    return (out.to(torch.float64).cpu().numpy(), lse.to(torch.float64).cpu().numpy(),
            opart.to(torch.float64).cpu().numpy(), err)


def half_ulp(ref, dtype: str):
    """Half a unit in the last place of ref in the output dtype (binary16: 11 significant
    bits, bfloat16: 8): the error of rounding the exact result once, which no kernel can avoid."""
    bits = 11 if dtype == "f16" else 8
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14 if dtype == "f16" else -126)   # subnormal spacing floor
    return np.where(a > 0, np.ldexp(1.0, (e - bits).astype(int)), 0.0)


def out_excess(out, ref, dtype: str) -> float:
    """max(|out - ref| - half_ulp(ref)): the output error beyond the final rounding.

    The bound for the final output is OUT_TOL on this excess. For the workloads'
    outputs (|o| well below 1) the half ulp is far below OUT_TOL, so this is the
    plain max |delta| <= 4e-3; it only matters for edge cases whose outputs reach
    |o| >= 1, where a bfloat16 output's own rounding (up to 2^-9 |o|) alone would
    exceed 4e-3.
    """
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(out - ref) - half_ulp(ref, dtype)
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isneginf(a) & np.isneginf(b)
    d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.nan_to_num(d, nan=np.inf).max()) if d.size else 0.0
