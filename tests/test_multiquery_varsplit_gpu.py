"""Several query tokens with per-sequence split counts (decode_attn_splitkv_multiquery_varsplit),
and large ragged batches with per-sequence split counts, against the float64 oracle."""
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


def run_mqv(p, tq, split_len, max_splits, tensors=None):
    q, k, v, cu = tensors if tensors is not None else to_device(p)
    q = q.view(p.B, tq, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * tq, p.Hq, p.D, max_splits)
    out = torch.empty(p.B, tq, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, ws, split_len=split_len,
                                               max_splits=max_splits, scale=p.scale, layout=p.layout)
    err = da.decode_attn_splitkv_get_error(ws)
    lse, opart = da.workspace_views(ws, p.B * tq, p.Hq, p.D, max_splits)
    return (out.to(torch.float64).cpu().numpy(),
            lse.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, max_splits),
            opart.to(torch.float64).cpu().numpy().reshape(p.B, tq, p.Hq, max_splits, p.D), err)


def check_mqv(p, tq, split_len, max_splits):
    out, lse, opart, err = run_mqv(p, tq, split_len, max_splits)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention_mq(p, tq)
    ref_op, ref_lse, sc = orc.split_partials_var_mq(p, tq, split_len, max_splits)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    for b in range(p.B):
        n = int(sc[b])
        if n == 1:
            continue   # the split step wrote the row itself; its workspace entries are not used
        assert np.array_equal(np.isneginf(lse[b, :, :, :n]), np.isneginf(ref_lse[b, :, :, :n])), b
        assert max_abs(lse[b, :, :, :n], ref_lse[b, :, :, :n]) <= LSE_TOL, b
        assert max_abs(opart[b, :, :, :n], ref_op[b, :, :, :n]) <= opart_tol(p), b


def nan_pad(p):
    """BHSD slabs past each sequence's length hold NaN, which no load may feed into a result."""
    for b, L in enumerate(p.lens):
        p.k[b, :, L:, :] = 0x7E00
        p.v[b, :, L:, :] = 0x7E00


CASES = [
    # name, B, tq, Hq, Hkv, D, lens, dtype, layout, split_len, max_splits, kv_rows
    # 28 columns per KV head (two 16-column chunks), ragged: the long sequences split, the
    # short ones stay whole (one of them shorter than the token count, one empty)
    ("qwen_g7_tq4", 6, 4, 28, 4, 128, [700, 5000, 3, 0, 2100, 64], "f16", LAYOUT_VARLEN, 512, 16, 0),
    ("llama_g4_tq2", 4, 2, 32, 8, 128, [1000, 5, 130, 4000], "bf16", LAYOUT_VARLEN, 256, 8, 0),
    ("mha_tq3_bhsd", 3, 3, 8, 8, 128, [300, 9, 1], "f16", LAYOUT_BHSD, 64, 8, 320),
    # 60 columns per KV head at head_dim 64: four chunks
    ("d64_g12_tq5", 5, 5, 12, 1, 64, [70, 1, 260, 129, 0], "bf16", LAYOUT_VARLEN, 64, 8, 0),
    ("tq16_one_seq", 1, 16, 16, 2, 128, [4096], "f16", LAYOUT_VARLEN, 1024, 8, 0),
    ("capped", 2, 2, 16, 2, 128, [3000, 200], "bf16", LAYOUT_VARLEN, 100, 5, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_multiquery_varsplit_parity(case):
    name, B, tq, Hq, Hkv, D, lens, dtype, layout, n, m, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, None, seed=zlib.crc32(name.encode()) % 983,
               kv_rows=kv_rows, tq=tq)
    if layout == LAYOUT_BHSD:
        nan_pad(p)
    check_mqv(p, tq, n, m)


def test_multiquery_varsplit_one_token_matches_varsplit_bit_for_bit():
    p = custom("mv1", 5, 28, 4, 128, [900, 64, 2000, 0, 3333], "f16", LAYOUT_VARLEN, None, seed=7)
    q, k, v, cu = to_device(p)
    a = run_mqv(p, 1, 512, 8, tensors=(q, k, v, cu))[0][:, 0]
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 8)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=512, max_splits=8, scale=p.scale)
    assert np.array_equal(a, out.to(torch.float64).cpu().numpy())


def test_multiquery_varsplit_equal_counts_match_uniform_bit_for_bit():
    """Ragged lengths that all get S_b = 4: the same bits as uniform splits with S = 4, although
    the uniform call hands out the sequences longest first and the per-sequence one in index
    order (an item's result does not depend on when it runs)."""
    p = custom("mvu", 4, 28, 4, 128, [1024, 1000, 900, 1020], "f16", LAYOUT_VARLEN, None, seed=8, tq=2)
    t = to_device(p)
    a = run_mqv(p, 2, 256, 4, tensors=t)[0]
    q, k, v, cu = t
    ws = da.alloc_workspace(p.B * 2, p.Hq, p.D, 4)
    out = torch.empty(p.B, 2, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_multiquery(q.view(p.B, 2, p.Hq, p.D), k, v, cu, out, ws, num_splits=4, scale=p.scale)
    assert np.array_equal(a, out.to(torch.float64).cpu().numpy())
    assert np.array_equal(a, run_mqv(p, 2, 256, 4, tensors=t)[0])   # and run to run


@pytest.mark.parametrize("B", [128, 129])
def test_varsplit_large_ragged_batch(B):
    """Per-sequence split counts over ragged batches of 128 and 129 sequences (their running split
    counts share the staged cu_seqlens_k area), lengths from a small set with empty and one-key
    sequences: every output element and every used partial against the oracle."""
    rng = np.random.default_rng(B + 1)
    lens = [int(x) for x in rng.choice([0, 1, 250, 500, 501, 1000, 1200], size=B)]
    p = custom(f"vord{B}", B, 8, 2, 64, lens, "bf16", LAYOUT_VARLEN, None, seed=B)
    q, k, v, cu = to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 8)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=250, max_splits=8, scale=p.scale)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    out = out.to(torch.float64).cpu().numpy()
    orc = oracle.default()
    ref, _ = orc.attention(p)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    lse, opart = da.workspace_views(ws, p.B, p.Hq, p.D, 8)
    lse, opart = lse.to(torch.float64).cpu().numpy(), opart.to(torch.float64).cpu().numpy()
    ref_op, ref_lse, sc = orc.split_partials_var(p, 250, 8)
    for b in range(p.B):
        n = int(sc[b])
        if n > 1:
            assert max_abs(lse[b, :, :n], ref_lse[b, :, :n]) <= LSE_TOL, b
            assert max_abs(opart[b, :, :n], ref_op[b, :, :n]) <= opart_tol(p), b


@pytest.mark.parametrize("B", [511, 512])
def test_varsplit_running_counts_in_and_out_of_the_staged_area(B):
    """Up to 511 sequences the per-sequence running split counts share the staged cu_seqlens_k
    area; from 512 they take an area of their own. Both sides of that limit, every output
    element against the oracle."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.choice([0, 1, 17, 64, 100, 300], size=B)]
    p = custom(f"vlim{B}", B, 4, 1, 64, lens, "f16", LAYOUT_VARLEN, None, seed=B)
    q, k, v, cu = to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 8)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=48, max_splits=8, scale=p.scale)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    ref, _ = oracle.default().attention(p)
    assert out_excess(out.to(torch.float64).cpu().numpy(), ref, p.dtype) <= OUT_TOL


def test_multiquery_varsplit_qwen_every_row():
    """The Qwen-shaped ragged batch with four query tokens, at the planner's split length (as the
    bench times it with --varsplit --tq 4): every (sequence, token, head) row against the oracle."""
    from synth.workloads import materialize, workload
    tq = 4
    p = workload("qwen_varlen", data=False)
    p.tq = tq
    materialize(p)
    n, m = da.varsplit_plan(p.B, p.Hq * tq, p.Hkv, p.D, p.total_kv, max(p.lens))
    out, lse, opart, err = run_mqv(p, tq, n, m)
    assert err == 0
    assert np.isfinite(out).all()
    ref, _ = oracle.default().attention_mq(p, tq)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL


def test_multiquery_varsplit_rejects_bad_arguments():
    p = custom("mvbad", 2, 8, 2, 64, [10, 20], "f16", LAYOUT_VARLEN, None, seed=9, tq=2)
    q, k, v, cu = to_device(p)
    q = q.view(p.B, 2, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * 2, p.Hq, p.D, 4)
    out = torch.empty(p.B, 2, p.Hq, p.D, dtype=torch.float16, device="cuda")
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, ws, split_len=0, max_splits=4)
    small = da.alloc_workspace(p.B, p.Hq, p.D, 4)   # rows for one token only
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, small, split_len=8, max_splits=4)


def test_multiquery_varsplit_cuda_graph_replay():
    """The call captured in a CUDA graph and replayed gives the eager call's bits (the work queue
    re-arms itself, nothing is allocated or copied on the host)."""
    p = custom("mvgraph", 3, 28, 4, 128, [3000, 100, 900], "f16", LAYOUT_VARLEN, None, seed=43, tq=4)
    q, k, v, cu = to_device(p)
    q = q.view(p.B, 4, p.Hq, p.D)
    ws = da.alloc_workspace(p.B * 4, p.Hq, p.D, 8)
    out = torch.empty(p.B, 4, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, ws, split_len=512, max_splits=8, scale=p.scale)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, ws, split_len=512, max_splits=8,
                                                   scale=p.scale)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert da.decode_attn_splitkv_get_error(ws) == 0
