"""The split step with CUDA-core FMA products (the comparison arm for the tensor-core
choice) against the float64 oracle: per-split lse and o, and the combined output."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_decoding_gb300 as da
from gpu_util import LSE_TOL, OUT_TOL, max_abs, opart_tol, out_excess, to_device, torch_dtype
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.load()


CASES = [
    # name, B, Hq, Hkv, D, lens, dtype, layout, S, kv_rows
    ("tiny_shape", 2, 4, 1, 64, [37, 200], "f16", LAYOUT_VARLEN, 4, 0),
    ("qwen_heads", 2, 28, 4, 128, [1000, 777], "f16", LAYOUT_VARLEN, 5, 0),
    ("mha_bhsd_nan_padded", 2, 32, 32, 128, [129, 250], "f16", LAYOUT_BHSD, 1, 256),
    ("llama_heads_bf16", 3, 32, 8, 128, [1024, 5, 333], "bf16", LAYOUT_VARLEN, 3, 0),
    ("codellama_heads", 2, 16, 2, 128, [700, 64], "f16", LAYOUT_VARLEN, 2, 0),
    ("empty_and_short", 4, 8, 2, 64, [0, 3, 17, 90], "bf16", LAYOUT_VARLEN, 6, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cuda_core_split_step_parity(case):
    name, B, Hq, Hkv, D, lens, dtype, layout, S, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, S, seed=zlib.crc32(name.encode()) % 983,
               kv_rows=kv_rows)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    q, k, v, cu = to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, S)
    da.decode_attn_splitkv_partial_cuda_core(q, k, v, cu, ws, num_splits=S, scale=p.scale, layout=p.layout)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    da.decode_attn_splitkv_combine(out, ws, num_splits=S)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    lse, opart = da.workspace_views(ws, p.B, p.Hq, p.D, S)
    lse = lse.to(torch.float64).cpu().numpy()
    opart = opart.to(torch.float64).cpu().numpy()
    orc = oracle.default()
    ref_op, ref_lse = orc.split_partials(p, S)
    ref, _ = orc.attention(p)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "empty-split pattern differs"
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)
    assert out_excess(out.to(torch.float64).cpu().numpy(), ref, p.dtype) <= OUT_TOL


def test_cuda_core_refuses_groups_over_eight():
    p = custom("g16", 1, 16, 1, 128, [100], "f16", LAYOUT_VARLEN, 1)
    q, k, v, cu = to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 1)
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_splitkv_partial_cuda_core(q, k, v, cu, ws, num_splits=1, scale=p.scale)
    assert e.value.status == da.DA_ERR_UNSUPPORTED
