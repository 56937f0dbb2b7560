"""Per-sequence split counts (decode_attn_splitkv_varsplit) vs the float64 oracle."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_decoding_gb300 as da
from gpu_util import LSE_TOL, OUT_TOL, max_abs, opart_tol, out_excess, to_device, torch_dtype
from oracle_pins import read_count_golden
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, custom, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.load()


def run_var(p, split_len, max_splits, tensors=None):
    q, k, v, cu = tensors if tensors is not None else to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, max_splits)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch_dtype(p), device="cuda")
    da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=split_len, max_splits=max_splits,
                                    scale=p.scale, layout=p.layout)
    err = da.decode_attn_splitkv_get_error(ws)
    lse, opart = da.workspace_views(ws, p.B, p.Hq, p.D, max_splits)
    return (out.to(torch.float64).cpu().numpy(), lse.to(torch.float64).cpu().numpy(),
            opart.to(torch.float64).cpu().numpy(), err)


def check_var(p, split_len, max_splits):
    out, lse, opart, err = run_var(p, split_len, max_splits)
    assert err == 0
    orc = oracle.default()
    ref, _ = orc.attention(p)
    ref_op, ref_lse, sc = orc.split_partials_var(p, split_len, max_splits)
    assert out_excess(out, ref, p.dtype) <= OUT_TOL
    for b in range(p.B):
        n = int(sc[b])
        assert max_abs(lse[b, :, :n], ref_lse[b, :, :n]) <= LSE_TOL, b
        assert max_abs(opart[b, :, :n], ref_op[b, :, :n]) <= opart_tol(p), b


CASES = [
    # name, B, Hq, Hkv, D, lens, dtype, layout, split_len, max_splits, kv_rows
    ("ragged_gqa7", 6, 28, 4, 128, [512, 8192, 1, 0, 3000, 777], "f16", LAYOUT_VARLEN, 512, 16, 0),
    ("short_splits", 3, 8, 1, 128, [100, 17, 64], "f16", LAYOUT_VARLEN, 16, 64, 0),
    ("capped", 2, 32, 8, 128, [4096, 300], "bf16", LAYOUT_VARLEN, 64, 5, 0),
    ("bhsd_mha", 3, 16, 16, 128, [900, 33, 450], "f16", LAYOUT_BHSD, 256, 8, 1000),
    ("d64_group12", 4, 12, 1, 64, [70, 1, 260, 129], "bf16", LAYOUT_VARLEN, 64, 8, 0),
    ("one_split_each", 3, 8, 2, 128, [50, 60, 70], "f16", LAYOUT_VARLEN, 4096, 4, 0),
    # 16 columns at head_dim 128: two n-tiles, with the per-sequence arrays in shared memory
    ("group16_d128", 3, 32, 2, 128, [2000, 5, 700], "f16", LAYOUT_VARLEN, 256, 8, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_varsplit_parity(case):
    name, B, Hq, Hkv, D, lens, dtype, layout, n, m, kv_rows = case
    p = custom(name, B, Hq, Hkv, D, lens, dtype, layout, None, seed=zlib.crc32(name.encode()) % 997,
               kv_rows=kv_rows)
    if layout == LAYOUT_BHSD:
        for b, L in enumerate(lens):
            p.k[b, :, L:, :] = 0x7E00
            p.v[b, :, L:, :] = 0x7E00
    check_var(p, n, m)


def test_varsplit_bounds_bit_exact_q_zero():
    """q = 0 pins every per-sequence split count and boundary: lse_s = ln(split length)."""
    for L, n, m, sb, bounds in read_count_golden():
        if L == 0:
            continue
        p = custom("cnt", 2, 4, 1, 64, [L, max(1, L // 3)], "f16", seed=9, q_std=0.0)
        out, lse, opart, err = run_var(p, n, m)
        assert err == 0
        for s in range(sb):
            ln = bounds[s + 1] - bounds[s]
            assert np.all(np.abs(lse[0, :, s] - math.log(ln)) <= 1e-5), (L, n, m, s)


def test_varsplit_qwen_workload_sampled():
    p = workload("qwen_varlen")
    n, m = da.varsplit_plan(p.B, p.Hq, p.Hkv, p.D, p.total_kv, max(p.lens))
    out, lse, opart, err = run_var(p, n, m)
    assert err == 0
    rng = np.random.default_rng(1)
    rb = rng.integers(0, p.B, 24).astype(np.int32)
    rh = rng.integers(0, p.Hq, 24).astype(np.int32)
    ref, ref_lse = oracle.default().attention_rows(p, rb, rh)
    assert max_abs(out[rb, rh], ref) <= OUT_TOL


def test_varsplit_deterministic_and_matches_uniform():
    p = custom("det", 4, 28, 4, 128, [5000, 700, 2000, 64], "f16", LAYOUT_VARLEN, None, seed=3)
    t = to_device(p)
    a = run_var(p, 512, 16, tensors=t)[0]
    b = run_var(p, 512, 16, tensors=t)[0]
    assert np.array_equal(a, b)
    # with every S_b equal to the uniform count, the two entry points agree bit for bit
    u = custom("uni", 2, 28, 4, 128, [1024, 1024], "f16", LAYOUT_VARLEN, None, seed=4)
    tu = to_device(u)
    vs = run_var(u, 256, 4, tensors=tu)[0]
    q, k, v, cu = tu
    ws = da.alloc_workspace(u.B, u.Hq, u.D, 4)
    out = torch.empty(u.B, u.Hq, u.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=4, scale=u.scale)
    assert np.array_equal(vs, out.to(torch.float64).cpu().numpy())


def test_varsplit_skewed_long_context_sampled():
    """One 128K sequence among short ones: per-sequence splits in the planner's configuration."""
    p = workload("llama_skewed")
    n, m = da.varsplit_plan(p.B, p.Hq, p.Hkv, p.D, p.total_kv, max(p.lens))
    out, lse, opart, err = run_var(p, n, m)
    assert err == 0
    rb = np.array([0, 0, 0, 1, 7, 15], dtype=np.int32)
    rh = np.array([0, 13, 31, 5, 20, 31], dtype=np.int32)
    ref, _ = oracle.default().attention_rows(p, rb, rh)
    assert max_abs(out[rb, rh], ref) <= OUT_TOL


def test_varsplit_bad_seqlens_flagged_and_contained():
    p = custom("vbad", 3, 8, 2, 128, [300, 400, 500], "f16", LAYOUT_VARLEN, None, seed=31)
    q, k, v, cu = to_device(p)
    cu_bad = cu.clone()
    cu_bad[3] = p.total_kv + 64
    out, lse, opart, err = run_var(p, 128, 8, tensors=(q, k, v, cu_bad))
    assert err & da.DA_DEVERR_SEQLENS
    ref, _ = oracle.default().attention(p)
    assert out_excess(out[:2], ref[:2], p.dtype) <= OUT_TOL
    assert not out[2].any()


def test_varsplit_cuda_graph_replay():
    p = custom("vgraph", 4, 28, 4, 128, [3000, 100, 900, 2500], "f16", LAYOUT_VARLEN, None, seed=32)
    q, k, v, cu = to_device(p)
    ws = da.alloc_workspace(p.B, p.Hq, p.D, 12)
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.float16, device="cuda")
    da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=256, max_splits=12, scale=p.scale)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=256, max_splits=12, scale=p.scale)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


_MIXED_MODES = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import split_kv_decode_decoding_gb300 as da
from gpu_util import to_device
from synth.workloads import LAYOUT_VARLEN, custom
da.load()
rng = np.random.default_rng(5)
p = custom("mixed", 600, 8, 2, 64, [int(x) for x in rng.integers(1, 40, 600)], "bf16", LAYOUT_VARLEN, None, seed=5)
q, k, v, cu = to_device(p)
ws = da.alloc_workspace(p.B, p.Hq, p.D, 4)
outs = []
for mode in ("var", "uniform", "var"):
    out = torch.empty(p.B, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    if mode == "var":
        da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=16, max_splits=3, scale=p.scale)
    else:
        da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=1, scale=p.scale)
    outs.append(out)
torch.cuda.synchronize()
assert da.decode_attn_splitkv_get_error(ws) == 0
assert torch.equal(outs[0], outs[2])
print("ok")
"""


def test_launch_configurations_of_one_kernel_mix_in_one_process():
    """One kernel launched with more shared memory (600 sequences with per-sequence splits: their
    running split counts need an area of their own), then less (uniform splits), then more again,
    in a fresh process: every launch succeeds and the repeated call gives the same bits."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _MIXED_MODES, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-2000:]
