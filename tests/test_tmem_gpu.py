"""The tcgen05 / tensor-memory comparison arm (decode_attn_splitkv_multiquery_tmem) against the
float64 oracle, per split and combined, and against the mma.sync path."""
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


def run(p, tq, S, fn):
    q, k, v, cu = to_device(p)
    q = q.view(p.B, tq, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * tq, p.Hq, p.D, S)
    out = torch.empty(p.B, tq, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    fn(q, k, v, cu, out, ws, num_splits=S, scale=p.scale, layout=p.layout)
    err = da.decode_attn_splitkv_get_error(ws)
    lse, opart = da.workspace_views(ws, p.B * tq, p.Hq, p.D, S)
    return (out.to(torch.float64).cpu().numpy(),
            lse.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S),
            opart.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S, p.D), err)


CASES = [
    # name, B, tq, Hq, Hkv, D, lens, dtype, layout, S, kv_rows
    ("qwen_g7_tq4", 2, 4, 28, 4, 128, [700, 64], "f16", LAYOUT_VARLEN, 3, 0),
    ("llama_g4_tq4_bf16", 3, 4, 32, 8, 128, [1000, 5, 130], "bf16", LAYOUT_VARLEN, 2, 0),
    ("bhsd_g4_tq5_nan_padded", 2, 5, 16, 4, 128, [500, 37], "bf16", LAYOUT_BHSD, 3, 512),
    ("d64_short_more_splits", 2, 3, 4, 1, 64, [2, 50], "f16", LAYOUT_VARLEN, 5, 0),
    ("g8_tq16_four_items", 1, 16, 16, 2, 128, [4096], "f16", LAYOUT_VARLEN, 8, 0),
    ("g20_one_token_direct", 2, 1, 20, 1, 128, [333, 1200], "f16", LAYOUT_VARLEN, 1, 0),
    ("g12_d64_bhsd_direct", 3, 2, 12, 1, 64, [64, 65, 190], "bf16", LAYOUT_BHSD, 1, 192),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tmem_parity(case):
    name, B, tq, Hq, Hkv, D, lens, dtype, layout, S, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, S, seed=zlib.crc32(name.encode()) % 997,
               kv_rows=kv_rows, tq=tq)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    out, lse, opart, err = run(p, tq, S, da.decode_attn_splitkv_multiquery_tmem)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    ref_op, ref_lse = orc.split_partials_mq(p, tq, S)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "empty-split pattern differs"
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)
    # the mma.sync path on the same inputs: the same result up to the order of the sums
    out2, lse2, _, err2 = run(p, tq, S, da.decode_attn_splitkv_multiquery)
    assert err2 == 0
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse2))
    assert max_abs(lse, lse2) <= 2 * LSE_TOL
    assert out_excess(out, out2, p.dtype) <= 2 * OUT_TOL


def test_tmem_ramping_scores_move_the_reference():
    """Scores climbing about 0.07 (log2 units) per key: each warp's lagging reference moves
    every couple of stages and O is rescaled in tensor memory; falling columns never move."""
    B, tq, Hq, Hkv, D, lens, S = 2, 2, 16, 2, 128, [1500, 700], 3
    p = custom("ramp_tmem", B, Hq, Hkv, D, lens, "f16", LAYOUT_VARLEN, S, seed=23, tq=tq)
    q = np.zeros((B, tq, Hq, D), np.float32)
    q[:, :, 0::2, :] = 0.25
    q[:, :, 1::2, :] = -0.25
    q[:, 1, :, :] *= 0.5
    p.q = q.astype(np.float16).view(np.uint16).reshape(p.q.shape)
    kf = np.zeros(p.k.shape, np.float32)
    for b, L in enumerate(lens):
        kf[p.cu[b]:p.cu[b] + L, :, :] = (np.arange(L) / 60.0).astype(np.float32)[:, None, None]
    p.k = kf.astype(np.float16).view(np.uint16)
    out, lse, opart, err = run(p, tq, S, da.decode_attn_splitkv_multiquery_tmem)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    ref_op, ref_lse = orc.split_partials_mq(p, tq, S)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)


def test_tmem_refuses_narrow_and_huge_groups():
    for Hq, Hkv, tq in ((8, 2, 2), (66, 1, 1)):
        p = custom("refuse", 1, Hq, Hkv, 64, [100], "f16", LAYOUT_VARLEN, 1, tq=tq)
        with pytest.raises(da.DecodeAttnError) as e:
            run(p, tq, 1, da.decode_attn_splitkv_multiquery_tmem)
        assert e.value.status == da.DA_ERR_UNSUPPORTED
