"""Several query tokens per sequence (decode_attn_splitkv_multiquery) vs the float64 oracle."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_decoding_gb300 as da
from gpu_util import LSE_TOL, OUT_TOL, max_abs, opart_tol, out_excess, to_device, torch_dtype
from oracle_pins import read_causal_golden
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.load()


def run_mq(p, tq, S, tensors=None):
    q, k, v, cu = tensors if tensors is not None else to_device(p)
    q = q.view(p.B, tq, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * tq, p.Hq, p.D, S)
    out = torch.empty(p.B, tq, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    da.decode_attn_splitkv_multiquery(q, k, v, cu, out, ws, num_splits=S, scale=p.scale,
                                      layout=p.layout)
    err = da.decode_attn_splitkv_get_error(ws)
    lse, opart = da.workspace_views(ws, p.B * tq, p.Hq, p.D, S)
    return (out.to(torch.float64).cpu().numpy(),
            lse.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S),
            opart.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S, p.D), err)


CASES = [
    # name, B, tq, Hq, Hkv, D, lens, dtype, layout, S, kv_rows
    ("llama_g4_tq2", 3, 2, 32, 8, 128, [1000, 5, 130], "bf16", LAYOUT_VARLEN, 4, 0),
    ("qwen_g7_tq4", 2, 4, 28, 4, 128, [700, 64], "f16", LAYOUT_VARLEN, 3, 0),
    ("mha_tq8_bhsd", 2, 8, 8, 8, 128, [300, 9], "f16", LAYOUT_BHSD, 2, 320),
    ("short_seq_more_splits", 2, 3, 4, 1, 64, [2, 50], "f16", LAYOUT_VARLEN, 5, 0),
    ("tq16_g8", 1, 16, 16, 2, 128, [4096], "f16", LAYOUT_VARLEN, 8, 0),
    ("one_split_direct", 3, 2, 8, 2, 64, [1, 2, 3], "bf16", LAYOUT_VARLEN, 1, 0),
    # 20 columns per KV head: a 16-column item and a 4-column one, over NaN-padded slabs
    ("bhsd_g4_tq5", 2, 5, 16, 4, 128, [500, 37], "bf16", LAYOUT_BHSD, 3, 512),
    # 16-column items at head_dim 128 whose columns see no key of a split: with 7 keys in 6
    # splits ([5, 7) the last), token 0 sees keys [0, 5) only, so its last split is empty
    # (lse -inf) while the item's other columns have keys
    ("d128_g4_tq3_unseen_split", 2, 3, 16, 4, 128, [7, 40], "bf16", LAYOUT_VARLEN, 6, 0),
    ("d128_g4_tq3_unseen_split_bhsd", 2, 3, 16, 4, 128, [7, 40], "f16", LAYOUT_BHSD, 6, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_multiquery_parity(case):
    name, B, tq, Hq, Hkv, D, lens, dtype, layout, S, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, S, seed=zlib.crc32(name.encode()) % 991,
               kv_rows=kv_rows, tq=tq)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    out, lse, opart, err = run_mq(p, tq, S)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    ref_op, ref_lse = orc.split_partials_mq(p, tq, S)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "empty-split pattern differs"
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)


def test_multiquery_causal_bounds_q_zero():
    """q = 0: lse = ln(keys the token sees in the split), -inf where it sees none (hand-worked)."""
    for L, tq, S, counts in read_causal_golden():
        p = custom("cz", 2, 4, 1, 64, [L, L + 3], "f16", seed=4, q_std=0.0, tq=tq)
        out, lse, opart, err = run_mq(p, tq, S)
        assert err == 0
        for t in range(tq):
            for s in range(S):
                n = counts[t][s]
                if n == 0:
                    assert np.isneginf(lse[0, t, :, s]).all()
                else:
                    assert np.abs(lse[0, t, :, s] - math.log(n)).max() <= 1e-5, (L, tq, S, t, s)


def test_multiquery_one_token_matches_single_query_bit_for_bit():
    p = custom("t1", 3, 28, 4, 128, [900, 64, 2000], "f16", LAYOUT_VARLEN, 4, seed=6)
    q, k, v, cu = to_device(p)
    a = run_mq(p, 1, 4, tensors=(q.view(p.B, 1, p.Hq, p.D), k, v, cu))[0][:, 0]
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 4)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=4, scale=p.scale)
    assert np.array_equal(a, out.to(torch.float64).cpu().numpy())


def test_multiquery_long_context_every_element():
    """Llama heads, 16 sequences of 32768 keys, two query tokens each (speculative decoding), at
    the picker's split count: every output row and every per-split partial against the oracle."""
    tq = 2
    p = custom("llama_S32768_B16_tq2", 16, 32, 8, 128, [32768] * 16, "bf16", LAYOUT_VARLEN, None,
               seed=0, tq=tq)
    S = da.num_splits(p.B, p.Hq * tq, p.Hkv, p.D, 32768, 32768)
    out, lse, opart, err = run_mq(p, tq, S)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    ref_op, ref_lse = orc.split_partials_mq(p, tq, S)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)


_MQ_REF = {}


def _mq_reference(name, tq):
    """The workload with tq query tokens and the oracle's output for it (shared by both arms)."""
    from synth.workloads import materialize, workload
    if (name, tq) not in _MQ_REF:
        p = workload(name, data=False)
        p.tq = tq
        materialize(p)
        ref, _ = oracle.default().attention_mq(p, tq)
        _MQ_REF[(name, tq)] = (p, ref)
    return _MQ_REF[(name, tq)]


@pytest.mark.parametrize("name,tq", [("qwen_varlen", 4), ("llama_S8192_B16", 4)])
@pytest.mark.parametrize("arm", ["mma_sync", "tmem"])
def test_multiquery_named_workloads_every_row(name, tq, arm):
    """Full-size workloads with several query tokens, the picker's split count (as the benchmark
    times them): every (sequence, token, head) row against the oracle, on both the default path
    and the tcgen05 arm; on the default path every per-split partial as well."""
    p, ref = _mq_reference(name, tq)
    S = da.num_splits(p.B, p.Hq * tq, p.Hkv, p.D, min(p.lens), max(p.lens))
    fn = da.decode_attn_splitkv_multiquery if arm == "mma_sync" else da.decode_attn_splitkv_multiquery_tmem
    q, k, v, cu = to_device(p)
    q = q.view(p.B, tq, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * tq, p.Hq, p.D, S)
    out = torch.empty(p.B, tq, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    fn(q, k, v, cu, out, ws, num_splits=S, scale=p.scale, layout=p.layout)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    out = out.to(torch.float64).cpu().numpy()
    assert np.isfinite(out).all()
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    if arm == "mma_sync":
        lse, opart = da.workspace_views(ws, p.B * tq, p.Hq, p.D, S)
        lse = lse.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S)
        opart = opart.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, S, p.D)
        ref_op, ref_lse = oracle.default().split_partials_mq(p, tq, S)
        assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
        assert max_abs(lse, ref_lse) <= LSE_TOL
        assert max_abs(opart, ref_op) <= opart_tol(p)


def test_multiquery_d64_bhsd_bf16():
    p = custom("mq64", 3, 12, 3, 64, [40, 3, 200], "bf16", LAYOUT_BHSD, 3, seed=41, kv_rows=210, tq=3)
    for b, L in enumerate(p.lens):
        p.k[b, :, L:, :] = 0x7E00
        p.v[b, :, L:, :] = 0x7E00
    out, lse, opart, err = run_mq(p, 3, 3)
    assert err == 0
    ref, _ = oracle.default().attention_mq(p, 3)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL


def test_multiquery_cuda_graph_replay():
    p = custom("mqg", 2, 16, 4, 128, [1000, 333], "f16", LAYOUT_VARLEN, 4, seed=42, tq=2)
    q, k, v, cu = to_device(p)
    q = q.view(p.B, 2, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * 2, p.Hq, p.D, 4)
    out = torch.empty(p.B, 2, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_multiquery(q, k, v, cu, out, ws, num_splits=4, scale=p.scale)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        da.decode_attn_splitkv_multiquery(q, k, v, cu, out, ws, num_splits=4, scale=p.scale)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("layout", [LAYOUT_VARLEN, LAYOUT_BHSD], ids=["varlen", "bhsd"])
def test_multiquery_ramping_scores(layout):
    """16-column items whose scores climb by about 0.07 (log2 units) per key: the running
    reference of the rising columns moves every couple of stages and the weights between
    moves reach 2^8; the other columns see falling scores and never move after the first box."""
    B, tq, Hq, Hkv, D, lens, S = 2, 2, 16, 2, 128, [1500, 700], 3
    p = custom("ramp", B, Hq, Hkv, D, lens, "f16", layout, S, seed=17, kv_rows=1536, tq=tq)
    q = np.zeros((B, tq, Hq, D), np.float32)
    q[:, :, 0::2, :] = 0.25
    q[:, :, 1::2, :] = -0.25
    q[:, 1, :, :] *= 0.5                      # the second token climbs at half the rate
    p.q = q.astype(np.float16).view(np.uint16).reshape(p.q.shape)
    kf = np.zeros(p.k.shape, np.float32)
    for b, L in enumerate(lens):
        ramp = (np.arange(L) / 60.0).astype(np.float32)   # scale * q.k_j = 2.83 * j / 60 at 0.25
        if layout == LAYOUT_BHSD:
            kf[b, :, :L, :] = ramp[None, :, None]
        else:
            kf[p.cu[b]:p.cu[b] + L, :, :] = ramp[:, None, None]
    p.k = kf.astype(np.float16).view(np.uint16)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    out, lse, opart, err = run_mq(p, tq, S)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    ref_op, ref_lse = orc.split_partials_mq(p, tq, S)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "empty-split pattern differs"
    assert max_abs(lse, ref_lse) <= LSE_TOL
    assert max_abs(opart, ref_op) <= opart_tol(p)
