"""CUDA path vs the float64 oracle, element by element, through the C ABI."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_decoding_gb300 as da
from gpu_util import LSE_TOL, OUT_TOL, max_abs, opart_tol, out_excess, run, to_device, torch_dtype
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, all_workload_names, custom, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.load()


def check_full(p, S):
    out, lse, opart, err = run(p, S)
    assert err == 0
    ref, _ = oracle.default().attention(p)
    ref_op, ref_lse = oracle.default().split_partials(p, S)
    e_out = out_excess(out, ref, p.dtype)
    e_lse = max_abs(lse, ref_lse)
    e_op = max_abs(opart, ref_op)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "empty-split pattern differs"
    assert e_out <= OUT_TOL, f"out max|d| {e_out}"
    assert e_lse <= LSE_TOL, f"lse_part max|d| {e_lse}"
    assert e_op <= opart_tol(p), f"o_part max|d| {e_op} > {opart_tol(p)}"
    return e_out, e_lse, e_op


def test_tiny_workload():
    p = workload("tiny")
    check_full(p, p.num_splits)


@pytest.mark.parametrize("R", [1, 8], ids=["one_head", "eight_packed_heads"])
def test_split_invariance_of_the_lecture_example(R):
    """The lecture page's exactness demonstration (04_flash_decoding.py, demo1_exact): one
    sequence of 10 000 keys, head_dim 128, 1 or 8 query heads packed on one KV head, split into
    1, 7, 64 and 1000 pieces: every split count against the same unsplit oracle result, and
    every per-split partial against the oracle's."""
    p = custom(f"demo1_R{R}", 1, R, 1, 128, [10000], "f16", LAYOUT_VARLEN, None, seed=11 + R)
    for S in (1, 7, 64, 1000):
        check_full(p, S)


CASES = [
    # name, B, Hq, Hkv, D, lens, dtype, layout, S, kv_rows
    ("short_tiles", 3, 8, 1, 128, [1, 16, 17], "f16", LAYOUT_VARLEN, 1, 0),
    ("stage_edges", 3, 8, 1, 128, [63, 64, 65], "f16", LAYOUT_VARLEN, 2, 0),
    ("qwen_heads", 2, 28, 4, 128, [1000, 777], "f16", LAYOUT_VARLEN, 7, 0),
    ("mha_bhsd", 2, 32, 32, 128, [300, 300], "f16", LAYOUT_BHSD, 3, 300),
    ("bhsd_padded", 2, 32, 32, 128, [129, 250], "f16", LAYOUT_BHSD, 4, 256),
    ("codellama_heads", 3, 16, 2, 128, [512, 100, 1023], "f16", LAYOUT_VARLEN, 16, 0),
    ("llama_heads_bf16", 2, 32, 8, 128, [1024, 555], "bf16", LAYOUT_VARLEN, 5, 0),
    ("group12_d64_bf16", 2, 12, 1, 64, [200, 333], "bf16", LAYOUT_VARLEN, 3, 0),
    ("group16", 2, 16, 1, 128, [80, 90], "f16", LAYOUT_VARLEN, 2, 0),
    ("empty_sequences", 4, 4, 4, 64, [0, 5, 0, 70], "f16", LAYOUT_VARLEN, 3, 0),
    ("more_splits_than_keys", 2, 8, 2, 64, [3, 10], "f16", LAYOUT_VARLEN, 6, 0),
    ("long_single_split", 1, 7, 1, 128, [4096], "f16", LAYOUT_VARLEN, 1, 0),
    ("d64_bhsd_bf16", 3, 8, 2, 64, [77, 1, 64], "bf16", LAYOUT_BHSD, 2, 80),
    ("many_splits", 2, 4, 1, 128, [2000, 1500], "f16", LAYOUT_VARLEN, 100, 0),
    # more than 8 columns per KV head: 16-column items (two n-tiles), and a second chunk
    ("group20_two_chunks", 2, 40, 2, 128, [300, 517], "f16", LAYOUT_VARLEN, 3, 0),
    ("group9_d64_bhsd", 2, 18, 2, 64, [100, 64], "bf16", LAYOUT_BHSD, 2, 128),
    # the shape of the MiniInfer page's self-test (flash_decode_splitk.py, __main__: fp16, batch 2,
    # 4 heads, head_dim 64, 256 keys, 4 splits, [batch, heads, seqlen, dim]), held here to the
    # oracle's tolerances rather than that test's 2e-2
    ("miniinfer_self_test_shape", 2, 4, 4, 64, [256, 256], "f16", LAYOUT_BHSD, 4, 256),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_cases(case):
    name, B, Hq, Hkv, D, lens, dtype, layout, S, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, S, seed=zlib.crc32(name.encode()) % 1000, kv_rows=kv_rows)
    if layout == LAYOUT_BHSD:
        # positions past each sequence's length hold NaN: they must never reach the result
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    check_full(p, S)


@pytest.mark.parametrize("B", [128, 129], ids=["sorted_128", "index_order_129"])
def test_ragged_batch_at_the_longest_first_limit(B):
    """Uniform splits over a ragged varlen batch: up to 128 sequences the split step hands them
    out longest first (ties by index), from 129 in index order. Lengths from a small set, so
    that many sequences tie, and a few empty ones; every element against the oracle."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.choice([0, 1, 33, 64, 65, 200, 513], size=B)]
    p = custom(f"rag{B}", B, 8, 2, 64, lens, "bf16", LAYOUT_VARLEN, 3, seed=B)
    check_full(p, 3)


def test_varlen_rows_past_the_last_sequence_are_ignored():
    p = custom("tailnan", 2, 8, 2, 128, [70, 45], "f16", LAYOUT_VARLEN, 3, seed=5, data=False)
    from synth.workloads import materialize
    materialize(p)
    cap = p.total_kv + 40
    k = np.full((cap, p.Hkv, p.D), 0x7E00, dtype=np.uint16)
    v = np.full((cap, p.Hkv, p.D), 0x7E00, dtype=np.uint16)
    k[: p.total_kv] = p.k
    v[: p.total_kv] = p.v
    p.k, p.v, p.kv_rows = k, v, cap
    check_full(p, 3)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 7, 9, 16, 37])
def test_split_bounds_bit_exact_q_zero(S):
    """q = 0: lse_s = ln(split length) exactly pins every split boundary on the device."""
    lens = [37, 200, 1, 16, 65, 129, 1000]
    p = custom("qz", len(lens), 4, 1, 64, lens, "f16", LAYOUT_VARLEN, S, seed=3, q_std=0.0)
    out, lse, opart, err = run(p, S)
    assert err == 0
    orc = oracle.default()
    for b, L in enumerate(lens):
        for s in range(S):
            lo, hi = orc.split_range(L, S, s)
            n = hi - lo
            for h in range(4):
                if n == 0:
                    assert lse[b, h, s] == -math.inf
                else:
                    assert abs(lse[b, h, s] - math.log(n)) <= 1e-5, (b, s, n, lse[b, h, s])
    ref_op, _ = orc.split_partials(p, S)
    assert max_abs(opart, ref_op) <= opart_tol(p)


@pytest.mark.parametrize("name", [n for n in all_workload_names() if n != "tiny"])
def test_named_workloads_every_element(name):
    """Full-size workloads in the launch configuration the benchmark uses (the picker's split
    count): every output row against the plain definition, and every per-split lse_s and o_s
    against the oracle's split partials at that split count."""
    p = workload(name)
    S = p.num_splits or da.num_splits(p.B, p.Hq, p.Hkv, p.D, min(p.lens), max(p.lens))
    out, lse, opart, err = run(p, S)
    assert err == 0
    orc = oracle.default()
    ref, ref_lse = orc.attention(p)
    e = max_abs(out, ref)
    assert e <= OUT_TOL, f"{name}: out max|d| {e}"
    ref_op, ref_lp = orc.split_partials(p, S)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lp)), "empty-split pattern differs"
    e_lse = max_abs(lse, ref_lp)
    assert e_lse <= LSE_TOL, f"{name}: lse_part max|d| {e_lse}"
    e_op = max_abs(opart, ref_op)
    assert e_op <= opart_tol(p), f"{name}: o_part max|d| {e_op} > {opart_tol(p)}"
    # the per-split log-sum-exps merge back to the row's total
    m = lse.max(axis=2, keepdims=True)
    tot = m[..., 0] + np.log(np.exp(lse - m).sum(axis=2))
    assert np.abs(tot - ref_lse).max() <= LSE_TOL


def _set_bits(p, name, values):
    """Round float values to the problem's dtype and store them as p.<name> bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch_dtype(p))
    setattr(p, name, t.view(torch.int16).numpy().view(np.uint16).reshape(getattr(p, name).shape))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", [LAYOUT_VARLEN, LAYOUT_BHSD], ids=["varlen", "bhsd"])
def test_single_token_ramping_scores(dtype, layout):
    """8-column items (one query token, G = 4) whose scores climb key after key: head 0 of
    each group by 0.068 and head 2 by 0.136 (log2 units) per key, so the running max moves on
    almost every 16-key box, in every warp and stage, and the accumulator is rescaled each time;
    heads 1 and 3 see falling scores and keep the first box's max. Every element of the output
    and of the per-split partials is checked."""
    B, Hq, Hkv, D, lens, S = 2, 8, 2, 128, [1500, 700], 3
    p = custom("ramp1", B, Hq, Hkv, D, lens, dtype, layout, S, seed=31, kv_rows=1536)
    q = np.zeros((B, Hq, D), np.float32)
    q[:, 0::4, :] = 0.25
    q[:, 1::4, :] = -0.25
    q[:, 2::4, :] = 0.5
    q[:, 3::4, :] = -0.5
    _set_bits(p, "q", q)
    kf = np.zeros(p.k.shape, np.float32)
    for b, L in enumerate(lens):
        ramp = (np.arange(L) / 60.0).astype(np.float32)   # scale * q.k_j = 2.83 * j / 60 at 0.25
        if layout == LAYOUT_BHSD:
            kf[b, :, :L, :] = ramp[None, :, None]
        else:
            kf[p.cu[b]:p.cu[b] + L, :, :] = ramp[:, None, None]
    _set_bits(p, "k", kf)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00 if dtype == "f16" else 0x7FC0
            p.v[b, :, L:, :] = 0x7E00 if dtype == "f16" else 0x7FC0
    check_full(p, S)


def _fp32_ulp(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    return np.ldexp(1.0, (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 23).astype(int))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", [LAYOUT_VARLEN, LAYOUT_BHSD], ids=["varlen", "bhsd"])
def test_single_token_one_key_dominates(dtype, layout):
    """One key scores more than 1000 above every other key of its sequence, late in a split
    (key 990 of [500, 1000), in the last stage's third warp): the heads that see it must return
    its value row, the others the ordinary softmax. The GPU twin of the oracle's one-hot pin.

    The split holding that key has lse_s near 1000, where one fp32 ulp is 2^-13: its bound is
    1e-4 plus 8 ulps of |lse| (the fp32 rounding of the score, of scale * log2 e folded into one
    constant, of the log2-domain sum and of the product by ln 2); every other value keeps the
    fixed bounds."""
    B, Hq, Hkv, D, lens, S = 2, 8, 2, 128, [1500, 700], 3
    p = custom("dom1", B, Hq, Hkv, D, lens, dtype, layout, S, seed=32, kv_rows=1536, k_std=0.25)
    q = np.zeros((B, Hq, D), np.float32)
    q[:, 0::2, :] = 4.0           # even heads: the planted key scores 4 * 23 * 128 / sqrt(128) = 1041
    q[:, 1::2, :] = -0.125        # odd heads: it scores -32, far below their usual keys
    _set_bits(p, "q", q)
    j = 990
    if layout == LAYOUT_BHSD:
        p.k[0, :, j, :] = 0x4DC0 if dtype == "f16" else 0x41B8   # 23.0
    else:
        p.k[p.cu[0] + j, :, :] = 0x4DC0 if dtype == "f16" else 0x41B8
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00 if dtype == "f16" else 0x7FC0
            p.v[b, :, L:, :] = 0x7E00 if dtype == "f16" else 0x7FC0
    out, lse, opart, err = run(p, S)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention(p)
    ref_op, ref_lp = orc.split_partials(p, S)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    # the even heads of sequence 0 return the planted key's value row
    from gpu_util import _decode
    vrow = _decode(p.v[0, :, j, :] if layout == LAYOUT_BHSD else p.v[p.cu[0] + j], dtype)   # [Hkv, D]
    for h in range(0, Hq, 2):
        assert np.abs(out[0, h] - vrow[h // (Hq // Hkv)]).max() <= OUT_TOL
    tol = LSE_TOL + 8 * _fp32_ulp(ref_lp)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lp))
    d = np.where(np.isneginf(ref_lp), 0.0, np.abs(lse - ref_lp))
    assert (d <= tol).all(), float((d - tol).max())
    assert max_abs(opart, ref_op) <= opart_tol(p)


def test_bad_seqlens_flagged_and_contained():
    p = custom("badcu", 3, 8, 2, 128, [50, 60, 70], "f16", LAYOUT_VARLEN, 2, seed=8)
    q, k, v, cu = to_device(p)
    cu_bad = cu.clone()
    cu_bad[3] = p.total_kv + 1000        # past the end of K/V
    out, lse, opart, err = run(p, 2, tensors=(q, k, v, cu_bad))
    assert err & da.DA_DEVERR_SEQLENS
    ref, _ = oracle.default().attention(p)
    assert max_abs(out[:2], ref[:2]) <= OUT_TOL
    assert not out[2].any() and np.isneginf(lse[2]).all()


def test_timeout_path_sets_flag_and_device_survives():
    ws = da.alloc_workspace(1, 1, 64, 1)
    da.decode_attn_splitkv_selftest_timeout(ws, 20_000)
    assert da.decode_attn_splitkv_get_error(ws) == da.DA_DEVERR_TIMEOUT
    assert da.decode_attn_splitkv_get_error(ws) == 0
    # the C reader returns DA_ERR_DEVICE_TIMEOUT for a timed-out wait, DA_OK otherwise
    import ctypes
    lib = da.load()
    bits = ctypes.c_uint32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    da.decode_attn_splitkv_selftest_timeout(ws, 20_000)
    assert lib.decode_attn_splitkv_get_error(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(bits),
                                             stream) == da.DA_ERR_DEVICE_TIMEOUT
    assert bits.value == da.DA_DEVERR_TIMEOUT
    assert lib.decode_attn_splitkv_get_error(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(bits),
                                             stream) == da.DA_OK
    assert bits.value == 0
    check_full(workload("tiny"), 4)


def test_partial_plus_combine_equals_full_and_is_deterministic():
    p = custom("det", 2, 28, 4, 128, [900, 1300], "f16", LAYOUT_VARLEN, 6, seed=12)
    q, k, v, cu = to_device(p)
    S = 6
    ws = da.alloc_workspace(p.B, p.Hq, p.D, S)
    a = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    b = torch.empty_like(a)
    da.decode_attn_splitkv(q, k, v, cu, a, ws, num_splits=S, scale=p.scale)
    da.decode_attn_splitkv_partial(q, k, v, cu, ws, num_splits=S, scale=p.scale)
    da.decode_attn_splitkv_combine(b, ws, num_splits=S)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    c = torch.empty_like(a)
    da.decode_attn_splitkv(q, k, v, cu, c, ws, num_splits=S, scale=p.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_cuda_graph_capture_and_side_stream():
    p = custom("graph", 4, 32, 8, 128, [700, 20, 1500, 333], "bf16", LAYOUT_VARLEN, 8, seed=13)
    q, k, v, cu = to_device(p)
    S = 8
    side = torch.cuda.Stream()
    ws = da.alloc_workspace(p.B, p.Hq, p.D, S, stream=side)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale, stream=side)
    side.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    ref, _ = oracle.default().attention(p)
    assert max_abs(out.to(torch.float64).cpu().numpy(), ref) <= OUT_TOL


def test_large_batch_reads_cu_from_global_memory():
    """More than 1024 sequences: the split kernel reads cu_seqlens_k from global memory
    instead of staging it in shared memory."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 90, 1500)]
    p = custom("bigB", 1500, 8, 2, 64, lens, "f16", LAYOUT_VARLEN, 2, seed=21)
    check_full(p, 2)


def test_maximum_split_count_on_a_long_sequence():
    """num_splits = DA_MAX_SPLITS on 131072 keys: 128-key splits, and a combine over 1024
    partials per row (the combine kernel's widest reduction)."""
    p = custom("maxS", 1, 8, 2, 128, [131072], "bf16", LAYOUT_VARLEN, da.DA_MAX_SPLITS, seed=22)
    check_full(p, da.DA_MAX_SPLITS)


def test_empty_cache_without_kv_buffers():
    """kv_rows = 0: every sequence is empty, K/V may be NULL; out = 0, every lse = -inf."""
    B, Hq, D, S = 3, 8, 128, 2
    q = torch.randn(B, Hq, D, device="cuda").to(torch.float16)
    k = torch.empty(0, 2, D, dtype=torch.float16, device="cuda")
    v = torch.empty(0, 2, D, dtype=torch.float16, device="cuda")
    cu = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    ws = da.alloc_workspace(B, Hq, D, S)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S)
    assert da.decode_attn_splitkv_get_error(ws) == 0
    assert not out.any()
    lse, _ = da.workspace_views(ws, B, Hq, D, S)
    assert torch.isneginf(lse).all()
    # a non-empty sequence with no K/V behind it is flagged and stays empty
    cu2 = torch.tensor([0, 0, 5, 5], dtype=torch.int32, device="cuda")
    da.decode_attn_splitkv(q, k, v, cu2, out, ws, num_splits=S)
    assert da.decode_attn_splitkv_get_error(ws) & da.DA_DEVERR_SEQLENS
    assert not out.any()


def test_one_workspace_across_calls_of_every_kind():
    """One workspace, sized for the largest call, reused by calls of every kind in a row: uniform
    splits (ragged and even batches, so both queue orders), per-sequence counts, several query
    tokens, one split. The work queue must come back to zero after each call whatever its item
    count (the last take resets it); every output against the oracle."""
    orc = oracle.default()
    ragged = custom("reuse_r", 5, 28, 4, 128, [700, 3000, 65, 1, 1500], "f16", LAYOUT_VARLEN, None, seed=51)
    even = custom("reuse_e", 3, 16, 4, 128, [640, 640, 640], "f16", LAYOUT_VARLEN, None, seed=52)
    multi = custom("reuse_m", 2, 28, 4, 128, [900, 300], "f16", LAYOUT_VARLEN, None, seed=53, tq=4)
    ws = da.alloc_workspace(8 * 4, 28, 128, 16)
    for rep in range(2):
        for p, kind, arg in ((ragged, "uniform", 7), (even, "uniform", 3), (ragged, "var", 256),
                             (multi, "mq", 2), (even, "uniform", 1), (multi, "mqvar", 200), (ragged, "uniform", 16)):
            q, k, v, cu = to_device(p)
            tq = p.tq
            out = torch.empty(p.B, tq, p.Hq, p.D, dtype=torch.float16, device="cuda")
            if kind == "uniform":
                da.decode_attn_splitkv(q, k, v, cu, out.view(p.B, p.Hq, p.D), ws, num_splits=arg, scale=p.scale)
            elif kind == "var":
                da.decode_attn_splitkv_varsplit(q, k, v, cu, out.view(p.B, p.Hq, p.D), ws, split_len=arg,
                                                max_splits=16, scale=p.scale)
            elif kind == "mq":
                da.decode_attn_splitkv_multiquery(q.view(p.B, tq, p.Hq, p.D), k, v, cu, out, ws, num_splits=arg,
                                                  scale=p.scale)
            else:
                da.decode_attn_splitkv_multiquery_varsplit(q.view(p.B, tq, p.Hq, p.D), k, v, cu, out, ws,
                                                           split_len=arg, max_splits=16, scale=p.scale)
            assert da.decode_attn_splitkv_get_error(ws) == 0, (rep, kind)
            ref = orc.attention_mq(p, tq)[0] if tq > 1 else orc.attention(p)[0][:, None]
            got = out.to(torch.float64).cpu().numpy()
            assert out_excess(got, ref, p.dtype) <= OUT_TOL, (rep, kind, arg)
