"""The no-allocation entry point against the workspace entry point.

decode_attn_splitkv_noalloc exists for callers that cannot allocate device
memory -- code behind a plugin interface that only hands it input and output
buffers, or a latency-critical path where cudaMalloc's device-wide
synchronisation is not allowed. It runs the same kernels on a scratch array
compiled into the library. This file is collected last on purpose, and works
both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_decoding_gb300 as da
from gpu_util import OUT_TOL, out_excess, to_device, torch_dtype
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.load()


def with_workspace(p, S, tensors):
    q, k, v, cu = tensors
    ws = da.alloc_workspace(p.B, p.Hq, p.D, S)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale, layout=p.layout)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    return out


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    a = custom("na_a", 4, 28, 4, 128, [700, 1500, 64, 3000], "f16", LAYOUT_VARLEN, 6, seed=71)
    b = custom("na_b", 3, 32, 8, 128, [2048, 333, 1024], "bf16", LAYOUT_BHSD, 9, seed=72,
               kv_rows=2048)
    ta, tb = to_device(a), to_device(b)
    ref_a = with_workspace(a, 6, ta)
    ref_b = with_workspace(b, 9, tb)
    out_a = torch.full_like(ref_a, float("nan"))
    out_b = torch.full_like(ref_b, float("nan"))
    # two calls back to back on the same stream; the second reuses the scratch the first left
    da.decode_attn_splitkv_noalloc(*ta, out_a, num_splits=6, scale=a.scale, layout=a.layout)
    da.decode_attn_splitkv_noalloc(*tb, out_b, num_splits=9, scale=b.scale, layout=b.layout)
    torch.cuda.synchronize()
    for got, ref in ((out_a, ref_a), (out_b, ref_b)):
        d = (got.double() - ref.double()).abs().max().item()
        assert d <= OUT_TOL, d
    # and once more with the first problem, after the second problem's contents
    again = torch.full_like(ref_a, float("nan"))
    da.decode_attn_splitkv_noalloc(*ta, again, num_splits=6, scale=a.scale, layout=a.layout)
    torch.cuda.synchronize()
    assert (again.double() - ref_a.double()).abs().max().item() <= OUT_TOL
    # and against the float64 oracle directly
    for p, got in ((a, again), (b, out_b)):
        ref, _ = oracle.default().attention(p)
        assert out_excess(got.double().cpu().numpy(), ref, p.dtype) <= OUT_TOL
    assert da.decode_attn_splitkv_noalloc_get_error() == 0


@pytest.mark.parametrize("case", [
    # head_dim 64 (four CTAs per SM, two heads per merge pass), several splits
    ("na_d64", 3, 12, 2, 64, [300, 17, 1024], "bf16", LAYOUT_VARLEN, 5, 0),
    # one split: the split kernel writes the output itself and no combine runs
    ("na_one_split", 4, 32, 8, 128, [512, 3, 2000, 64], "f16", LAYOUT_VARLEN, 1, 0),
    ("na_one_split_d64_bhsd", 2, 8, 8, 64, [100, 37], "f16", LAYOUT_BHSD, 1, 128),
], ids=lambda c: c[0])
def test_noalloc_head_dim_64_and_single_split(case):
    name, B, Hq, Hkv, D, lens, dtype, layout, S, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, S, seed=len(name), kv_rows=kv_rows)
    t = to_device(p)
    ref_ws = with_workspace(p, S, t)
    out = torch.full_like(ref_ws, float("nan"))
    da.decode_attn_splitkv_noalloc(*t, out, num_splits=S, scale=p.scale, layout=p.layout)
    torch.cuda.synchronize()
    assert (out.double() - ref_ws.double()).abs().max().item() <= OUT_TOL
    ref, _ = oracle.default().attention(p)
    assert out_excess(out.double().cpu().numpy(), ref, p.dtype) <= OUT_TOL
    assert da.decode_attn_splitkv_noalloc_get_error() == 0


def test_noalloc_reports_device_errors_through_its_reader():
    """A cu_seqlens_k entry past the end of K/V sets DA_DEVERR_SEQLENS in the scratch array's
    error word; the reader returns it once, and the next good call starts clean."""
    p = custom("na_badcu", 3, 8, 2, 128, [50, 60, 70], "f16", LAYOUT_VARLEN, 2, seed=9)
    q, k, v, cu = to_device(p)
    bad = cu.clone()
    bad[3] = p.total_kv + 1000
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_noalloc(q, k, v, bad, out, num_splits=2, scale=p.scale)
    assert da.decode_attn_splitkv_noalloc_get_error() == da.DA_DEVERR_SEQLENS
    assert da.decode_attn_splitkv_noalloc_get_error() == 0
    ref, _ = oracle.default().attention(p)
    got = out.double().cpu().numpy()
    assert out_excess(got[:2], ref[:2], p.dtype) <= OUT_TOL and not got[2].any()
    da.decode_attn_splitkv_noalloc(q, k, v, cu, out, num_splits=2, scale=p.scale)
    assert da.decode_attn_splitkv_noalloc_get_error() == 0
    assert out_excess(out.double().cpu().numpy(), ref, p.dtype) <= OUT_TOL


def test_noalloc_refuses_problems_beyond_its_scratch():
    p = custom("na_big", 64, 28, 4, 128, [16] * 64, "f16", LAYOUT_VARLEN, 16, seed=73)
    need = da.workspace_size(p.B, p.Hq, p.D, 16)
    assert need > da.DA_NOALLOC_SCRATCH_BYTES
    q, k, v, cu = to_device(p)
    out = torch.zeros(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_splitkv_noalloc(q, k, v, cu, out, num_splits=16, scale=p.scale)
    assert e.value.status == da.DA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert not out.any()
