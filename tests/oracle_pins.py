"""Pins for the float64 oracle: checks against what the pages and the mathematics fix.

Each pin takes an ``oracle.Oracle`` so that tests/test_oracle.py can run them on
the real oracle (all must pass) and tests/test_oracle_mutants.py on copies with
a planted mistake (at least one must fail). None of them re-types the oracle's
general formula: they use closed forms for special inputs, hand-worked values,
invariants, and library routines (numpy, torch) as an independent third
implementation.

Sources of the facts pinned here:
* proportional split bounds: TileLang decode_attention_splitkv.py, split segment;
* split + log-sum-exp merge equals the unsplit result, for 1/7/64/1000 splits,
  1 or 8 packed heads: CS349E lecture 11 04_flash_decoding.py, demo1_exact;
* GQA packing equals per-head attention with K/V repeated: the same lecture,
  demo1_exact second observation and demo3_vs_blog (eager copies K/V per head);
* softmax(q k^T * scale) @ V: MiniInfer flash_decode_splitk.py,
  flash_decode_reference;
* empty split -> weight 0 (m = -inf, l = 0): MiniInfer _splitk_reduce_kernel.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from synth import round_bf16, round_f16
from synth.workloads import LAYOUT_BHSD, LAYOUT_VARLEN, custom

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _decode_all(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Library decode (torch views), independent of the oracle's decoder."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.to(torch.float64).numpy()


def read_split_golden():
    rows = []
    with open(os.path.join(GOLDEN, "split_bounds.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals = [int(x) for x in line.split()]
            rows.append((vals[0], vals[1], vals[2:]))
    return rows


# ---------------------------------------------------------------- encodings
def pin_f16_decoder(o):
    known = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
             0x0400: 2.0 ** -14, 0x3555: 0.333251953125, 0x3800: 0.5, 0x4248: 3.140625}
    for bits, val in known.items():
        assert o.f16_to_double(bits) == val, hex(bits)
    assert math.isinf(o.f16_to_double(0x7C00)) and math.isnan(o.f16_to_double(0x7E00))
    allbits = np.arange(65536, dtype=np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_double(int(b)) for b in allbits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def pin_bf16_decoder(o):
    known = {0x3F80: 1.0, 0x4049: 3.140625, 0xC2F7: -123.5, 0x0001: 2.0 ** -133,
             0x0080: 2.0 ** -126, 0x7F7F: float(torch.finfo(torch.bfloat16).max)}
    for bits, val in known.items():
        assert o.bf16_to_double(bits) == val, hex(bits)
    allbits = np.arange(65536, dtype=np.uint16)
    ref = _decode_all(allbits, "bf16")
    got = np.array([o.bf16_to_double(int(b)) for b in allbits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ------------------------------------------------------------- split bounds
def pin_split_bounds_golden(o):
    for L, S, bounds in read_split_golden():
        assert len(bounds) == S + 1
        for s in range(S):
            assert o.split_range(L, S, s) == (bounds[s], bounds[s + 1]), (L, S, s)


def pin_split_bounds_partition(o):
    for L in list(range(0, 70)) + [255, 256, 257, 4096, 131072, 2_000_000_000]:
        for S in (1, 2, 3, 4, 5, 7, 8, 16, 64, 152, 1000):
            prev = 0
            lo_len, hi_len = L // S, -(-L // S)
            for s in range(S):
                a, b = o.split_range(L, S, s)
                assert a == prev and b >= a
                assert lo_len <= b - a <= hi_len
                if S <= L:
                    assert b > a
                prev = b
            assert prev == L


# -------------------------------------------------------- attention pins
def _dec(p, bits):
    return _decode_all(bits, p.dtype)


def pin_split_invariance(o):
    """demo1_exact: L = 10000, D = 128, R in {1, 8} packed heads, S in {1, 7, 64, 1000}."""
    for R in (1, 8):
        p = custom("inv", 1, R, 1, 128, [10000], "f16", seed=7)
        ref, ref_lse = o.attention(p)
        for S in (1, 7, 64, 1000):
            op, lp = o.split_partials(p, S)
            out, lse = o.merge(op, lp)
            assert np.abs(out - ref).max() <= 1e-12, (R, S)
            assert np.abs(lse - ref_lse).max() <= 1e-12, (R, S)


def pin_weights_sum_to_one(o):
    p = custom("w", 3, 4, 2, 64, [1, 50, 333], "f16", seed=3)
    for b in range(3):
        for h in range(4):
            w = o.weights(p, b, h)
            assert w.size == p.lens[b]
            assert (w >= 0).all()
            assert abs(w.sum() - 1.0) <= 1e-14
    pb = custom("wb", 2, 2, 1, 64, [40, 9], "bf16", seed=5)
    assert abs(o.weights(pb, 0, 1).sum() - 1.0) <= 1e-14


def pin_single_key(o):
    """A single key gets all the weight: out = v_0 exactly, for every head."""
    p = custom("one", 3, 6, 2, 64, [1, 1, 1], "f16", seed=11)
    out, _ = o.attention(p)
    v = _dec(p, p.v)
    for b in range(3):
        for h in range(6):
            assert np.array_equal(out[b, h], v[b, h // 3]), (b, h)


def pin_single_key_lse(o):
    """q = e_0, k_0 = 2 e_0, scale 1/2: the only score is 1, so lse = 1."""
    p = custom("lse1", 1, 1, 1, 4, [1], "f16", scale=0.5, data=True)
    p.q[...] = 0
    p.k[...] = 0
    p.q[0, 0, 0] = round_f16(1.0)
    p.k[0, 0, 0] = round_f16(2.0)
    out, lse = o.attention(p)
    assert lse[0, 0] == 1.0
    _, lp = o.split_partials(p, 1)
    assert lp[0, 0, 0] == 1.0


def pin_constant_v(o):
    for dtype in ("f16", "bf16"):
        p = custom("cv", 2, 4, 2, 64, [17, 300], dtype, seed=2, v_mean=0.75, v_std=0.0)
        out, _ = o.attention(p)
        assert np.abs(out - 0.75).max() <= 1e-14
        op, lp = o.split_partials(p, 5)
        assert np.abs(op - 0.75).max() <= 1e-14


def pin_gqa_packing(o):
    """GQA with 8 query heads on 2 KV heads equals 8 independent heads with K/V repeated."""
    p = custom("gqa", 3, 8, 2, 64, [5, 64, 129], "f16", seed=9)
    ref, ref_lse = o.attention(p)
    m = custom("mha", 3, 8, 8, 64, [5, 64, 129], "f16", data=False)
    m.cu = p.cu.copy()
    m.kv_rows = p.kv_rows
    m.q = p.q.copy()
    m.k = np.repeat(p.k, 4, axis=1).copy()
    m.v = np.repeat(p.v, 4, axis=1).copy()
    out, lse = o.attention(m)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def pin_hand_example(o):
    """scale 1, q = (1, 0); scores 0, 1, 2; v = (1,0), (0,1), (1,1).

    Worked by hand: Z = 1 + e + e^2, out = ((1 + e^2)/Z, (e + e^2)/Z), lse = ln Z.
    Two splits: [0,1) and [1,3). Split 0: lse = 0, o = (1, 0). Split 1:
    lse = ln(e + e^2) = 1 + ln(1 + e), o = (e/(1 + e), 1).
    """
    p = custom("hand", 1, 1, 1, 2, [3], "f16", scale=1.0)
    one = round_f16(1.0)
    p.q[...] = 0
    p.q[0, 0, 0] = one
    p.k[...] = 0
    p.k[1, 0, 0] = one
    p.k[2, 0, 0] = round_f16(2.0)
    p.v[...] = 0
    p.v[0, 0, 0] = one
    p.v[1, 0, 1] = one
    p.v[2, 0, :] = one
    e = math.e
    Z = 1 + e + e * e
    out, lse = o.attention(p)
    assert abs(out[0, 0, 0] - (1 + e * e) / Z) <= 1e-15
    assert abs(out[0, 0, 1] - (e + e * e) / Z) <= 1e-15
    assert abs(lse[0, 0] - math.log(Z)) <= 1e-15
    op, lp = o.split_partials(p, 2)
    assert lp[0, 0, 0] == 0.0 and np.array_equal(op[0, 0, 0], [1.0, 0.0])
    assert abs(lp[0, 0, 1] - (1 + math.log1p(e))) <= 1e-15
    assert abs(op[0, 0, 1, 0] - e / (1 + e)) <= 1e-15 and abs(op[0, 0, 1, 1] - 1.0) <= 1e-15


def pin_q_zero_closed_form(o):
    """q = 0: every score is 0, so lse_s = ln(split length) and o_s = mean of V over the split.

    For the tiny workload (lengths 37 and 200, 4 splits) the split lengths come
    from the golden bounds: 9, 9, 9, 10 and 50, 50, 50, 50.
    """
    p = custom("qz", 2, 4, 1, 64, [37, 200], "f16", seed=0, q_std=0.0)
    assert not p.q.any()
    op, lp = o.split_partials(p, 4)
    v = _dec(p, p.v)
    golden = {L: b for L, S, b in read_split_golden() if S == 4}
    for bi, L in enumerate((37, 200)):
        bounds = golden[L]
        base = int(p.cu[bi])
        for s in range(4):
            n = bounds[s + 1] - bounds[s]
            mean = v[base + bounds[s]: base + bounds[s + 1], 0, :].mean(axis=0)
            for h in range(4):
                assert abs(lp[bi, h, s] - math.log(n)) <= 1e-13
                assert np.abs(op[bi, h, s] - mean).max() <= 1e-14
    out, lse = o.attention(p)
    for bi, L in enumerate((37, 200)):
        mean = v[int(p.cu[bi]): int(p.cu[bi + 1]), 0, :].mean(axis=0)
        assert np.abs(out[bi] - mean).max() <= 1e-14
        assert np.abs(lse[bi] - math.log(L)).max() <= 1e-13


def pin_one_hot_dominance(o):
    """One key scores 1024 above the rest: its value comes back (needs the max subtracted)."""
    p = custom("dom", 1, 1, 1, 8, [40], "f16", scale=1.0, seed=4)
    p.q[...] = 0
    p.q[0, 0, 0] = round_f16(32.0)
    p.k[:, :, 0] = 0
    p.k[23, 0, 0] = round_f16(32.0)
    out, lse = o.attention(p)
    v = _dec(p, p.v)
    assert np.abs(out[0, 0] - v[23, 0]).max() <= 1e-12
    assert abs(lse[0, 0] - 1024.0) <= 1e-9
    op, lp = o.split_partials(p, 3)
    m, ml = o.merge(op, lp)
    assert np.abs(m[0, 0] - v[23, 0]).max() <= 1e-12


def _torch_attention(p):
    """Library cross-check: float64 torch softmax attention, one (b, h) at a time."""
    q = torch.from_numpy(_dec(p, p.q))
    k = torch.from_numpy(_dec(p, p.k))
    v = torch.from_numpy(_dec(p, p.v))
    G = p.Hq // p.Hkv
    out = torch.zeros(p.B, p.Hq, p.D, dtype=torch.float64)
    lse = torch.full((p.B, p.Hq), -math.inf, dtype=torch.float64)
    for b in range(p.B):
        L = int(p.cu[b + 1] - p.cu[b])
        if L == 0:
            continue
        for h in range(p.Hq):
            if p.layout == LAYOUT_VARLEN:
                kk = k[int(p.cu[b]): int(p.cu[b + 1]), h // G, :]
                vv = v[int(p.cu[b]): int(p.cu[b + 1]), h // G, :]
            else:
                kk = k[b, h // G, :L, :]
                vv = v[b, h // G, :L, :]
            sc = (kk @ q[b, h]) * p.scale
            out[b, h] = torch.softmax(sc, dim=0) @ vv
            lse[b, h] = torch.logsumexp(sc, dim=0)
    return out.numpy(), lse.numpy()


def pin_library_cross_check(o):
    cases = [
        custom("x1", 3, 6, 2, 64, [1, 17, 130], "f16", seed=21),
        custom("x2", 2, 7, 1, 128, [300, 45], "f16", seed=22),
        custom("x3", 2, 4, 4, 128, [64, 65], "bf16", seed=23),
        custom("x4", 2, 8, 2, 64, [33, 96], "f16", layout=LAYOUT_BHSD, kv_rows=100, seed=24),
        custom("x5", 2, 2, 1, 64, [0, 12], "bf16", seed=25),
    ]
    for p in cases:
        ref, ref_lse = _torch_attention(p)
        out, lse = o.attention(p)
        assert np.abs(out - ref).max() <= 1e-12, p.name
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12, p.name


def pin_bhsd_matches_varlen(o):
    """The same cache in both layouts gives identical results; BHSD padding rows are never read."""
    lens = [5, 40, 17]
    vl = custom("vl", 3, 4, 2, 64, lens, "f16", seed=31)
    cap = 48
    bh = custom("bh", 3, 4, 2, 64, lens, "f16", layout=LAYOUT_BHSD, kv_rows=cap, data=False)
    bh.q, bh.cu, bh.kv_rows = vl.q.copy(), vl.cu.copy(), cap
    nan = np.uint16(0x7E00)
    bh.k = np.full((3, 2, cap, 64), nan, dtype=np.uint16)
    bh.v = np.full((3, 2, cap, 64), nan, dtype=np.uint16)
    for b, L in enumerate(lens):
        rows = slice(int(vl.cu[b]), int(vl.cu[b + 1]))
        bh.k[b, :, :L, :] = vl.k[rows].transpose(1, 0, 2)
        bh.v[b, :, :L, :] = vl.v[rows].transpose(1, 0, 2)
    a, la = o.attention(vl)
    c, lc = o.attention(bh)
    assert np.array_equal(a, c) and np.array_equal(la, lc)
    pa, pla = o.split_partials(vl, 6)
    pc, plc = o.split_partials(bh, 6)
    assert np.array_equal(pa, pc) and np.array_equal(pla, plc)


def pin_empty_splits_and_sequences(o):
    p = custom("emp", 3, 2, 1, 64, [3, 0, 9], "f16", seed=41)
    ref, ref_lse = o.attention(p)
    assert not ref[1].any() and np.all(np.isneginf(ref_lse[1]))
    S = 5
    op, lp = o.split_partials(p, S)
    # sequence 0 (3 keys, 5 splits): splits 0 and 2 are empty
    assert np.isneginf(lp[0, :, 0]).all() and np.isneginf(lp[0, :, 2]).all()
    assert not op[0, :, 0].any() and not op[0, :, 2].any()
    assert np.isfinite(lp[0, :, 1]).all() and np.isfinite(lp[0, :, 3]).all()
    assert np.isneginf(lp[1]).all() and not op[1].any()
    out, lse = o.merge(op, lp)
    assert np.abs(out - ref).max() <= 1e-12
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))


def pin_threads_deterministic(o):
    p = custom("thr", 4, 8, 2, 64, [100, 7, 55, 300], "bf16", seed=51)
    a, la = o.attention(p, nthreads=1)
    b, lb = o.attention(p, nthreads=5)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def pin_rows_match_full(o):
    p = custom("rows", 3, 6, 3, 64, [20, 200, 77], "f16", seed=61)
    full, full_lse = o.attention(p)
    rb = np.array([0, 2, 1, 2], dtype=np.int32)
    rh = np.array([5, 0, 3, 4], dtype=np.int32)
    out, lse = o.attention_rows(p, rb, rh)
    assert np.array_equal(out, full[rb, rh]) and np.array_equal(lse, full_lse[rb, rh])


def pin_rows_mq_match_full(o):
    """The row selector for several query tokens (the checker of the full-size multi-token GPU
    tests) equals the whole-problem function at the same (b, t, h), bit for bit, in both
    layouts, for tokens after the first and for a token that sees no key."""
    for layout in (LAYOUT_VARLEN, LAYOUT_BHSD):
        tq = 4
        p = custom("rowsmq", 3, 4, 2, 64, [30, 5, 2], "bf16", layout=layout, seed=62, tq=tq,
                   kv_rows=32 if layout == LAYOUT_BHSD else 0)
        full, full_lse = o.attention_mq(p, tq)
        rb = np.array([0, 2, 1, 0, 1, 2, 0, 2], dtype=np.int32)
        rt = np.array([3, 1, 2, 1, 3, 0, 2, 3], dtype=np.int32)
        rh = np.array([0, 3, 1, 2, 2, 1, 3, 0], dtype=np.int32)
        out, lse = o.attention_rows_mq(p, tq, rb, rt, rh)
        assert np.array_equal(out, full[rb, rt, rh]), layout
        assert np.array_equal(lse, full_lse[rb, rt, rh]), layout
        # token 0 of the two-key sequence sees no key (position 2 - 4 + 0 < 0): out 0, lse -inf
        assert not out[5].any() and lse[5] == -math.inf


def read_count_golden():
    rows = []
    with open(os.path.join(GOLDEN, "split_counts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v = [int(x) for x in line.split()]
            rows.append((v[0], v[1], v[2], v[3], v[4:]))
    return rows


def pin_split_counts_golden(o):
    """Per-sequence split counts and bounds, pinned by q = 0: lse_s = ln(split length)."""
    for L, n, m, sb, bounds in read_count_golden():
        assert len(bounds) == sb + 1
        p = custom("cnt", 1, 2, 1, 64, [L], "f16", seed=5, q_std=0.0)
        op, lp, sc = o.split_partials_var(p, n, m)
        assert sc[0] == sb, (L, n, m)
        v = _dec(p, p.v)
        for s_ in range(m):
            if s_ < sb and bounds[s_ + 1] > bounds[s_]:
                ln = bounds[s_ + 1] - bounds[s_]
                assert abs(lp[0, 1, s_] - math.log(ln)) <= 1e-13, (L, n, m, s_)
                mean = v[bounds[s_]: bounds[s_ + 1], 0, :].mean(axis=0)
                assert np.abs(op[0, 1, s_] - mean).max() <= 1e-14
            else:
                assert lp[0, 1, s_] == -math.inf and not op[0, 1, s_].any()


def pin_varsplit_merge_invariance(o):
    """Per-sequence split counts merge back to the unsplit result (ragged batch, GQA)."""
    p = custom("vs", 5, 8, 2, 64, [1, 90, 1000, 333, 0], "f16", seed=17)
    ref, ref_lse = o.attention(p)
    for n, m in ((16, 64), (100, 4), (64, 1), (7, 200)):
        op, lp, sc = o.split_partials_var(p, n, m)
        out, lse = o.merge(op, lp)
        assert np.abs(out - ref).max() <= 1e-12, (n, m)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12
        for b, L in enumerate(p.lens):
            assert sc[b] == (1 if L == 0 else min(m, -(-L // n)))


def read_causal_golden():
    rows = []
    with open(os.path.join(GOLDEN, "causal_splits.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [x.split() for x in line.split("|")]
            L, tq, S = (int(x) for x in parts[0])
            rows.append((L, tq, S, [[int(x) for x in c] for c in parts[1:]]))
    return rows


def pin_mq_causal_counts_golden(o):
    """Several query tokens: q = 0 gives lse = ln(keys seen) per token and split (hand-worked)."""
    for L, tq, S, counts in read_causal_golden():
        assert len(counts) == tq and all(len(c) == S for c in counts)
        p = custom("cz", 1, 2, 1, 64, [L], "f16", seed=3, q_std=0.0, tq=tq)
        op, lp = o.split_partials_mq(p, tq, S)
        out, lse = o.attention_mq(p, tq)
        v = _dec(p, p.v)
        for t in range(tq):
            for s_ in range(S):
                n = counts[t][s_]
                if n == 0:
                    assert np.isneginf(lp[0, t, :, s_]).all() and not op[0, t, :, s_].any()
                else:
                    assert np.abs(lp[0, t, :, s_] - math.log(n)).max() <= 1e-13, (L, tq, S, t, s_)
            vis = sum(counts[t])
            if vis == 0:
                assert not out[0, t].any() and np.isneginf(lse[0, t]).all()
            else:
                assert np.abs(lse[0, t] - math.log(vis)).max() <= 1e-13
                assert np.abs(out[0, t] - v[:vis, 0, :].mean(axis=0)).max() <= 1e-14


def pin_mq_tq1_equals_single(o):
    p = custom("t1", 3, 8, 2, 64, [9, 100, 1], "bf16", seed=12)
    a, la = o.attention(p)
    b, lb = o.attention_mq(p, 1)
    assert np.array_equal(a, b[:, 0]) and np.array_equal(la, lb[:, 0])
    pa, pla = o.split_partials(p, 4)
    pb, plb = o.split_partials_mq(p, 1, 4)
    assert np.array_equal(pa, pb[:, 0]) and np.array_equal(pla, plb[:, 0])


def pin_mq_token_equals_truncated_single(o):
    """Token t equals a single-query problem whose cache stops at the token's own position."""
    for layout in (LAYOUT_VARLEN, LAYOUT_BHSD):
        lens = [40, 7, 3]
        tq = 4
        p = custom("mq", 3, 8, 2, 64, lens, "f16", layout=layout, seed=8, tq=tq,
                   kv_rows=48 if layout == LAYOUT_BHSD else 0)
        out, lse = o.attention_mq(p, tq)
        for b, L in enumerate(lens):
            for t in range(tq):
                vis = max(0, L - tq + t + 1)
                s1 = custom("one", 1, 8, 2, 64, [vis], "f16", data=False)
                s1.q = np.ascontiguousarray(p.q[b, t][None])
                if layout == LAYOUT_VARLEN:
                    s1.k = np.ascontiguousarray(p.k[p.cu[b]: p.cu[b] + vis])
                    s1.v = np.ascontiguousarray(p.v[p.cu[b]: p.cu[b] + vis])
                else:
                    s1.k = np.ascontiguousarray(p.k[b, :, :vis].transpose(1, 0, 2))
                    s1.v = np.ascontiguousarray(p.v[b, :, :vis].transpose(1, 0, 2))
                s1.cu = np.array([0, vis], dtype=np.int32)
                s1.kv_rows = vis
                ref, rl = o.attention(s1)
                assert np.array_equal(out[b, t], ref[0]), (layout, b, t)
                assert np.array_equal(lse[b, t], rl[0])


def pin_mq_split_invariance(o):
    p = custom("mqs", 2, 6, 3, 64, [300, 17], "f16", seed=14, tq=5)
    ref, ref_lse = o.attention_mq(p, 5)
    for S in (1, 3, 8, 40):
        op, lp = o.split_partials_mq(p, 5, S)
        out, lse = o.merge(op, lp)
        assert np.abs(out - ref).max() <= 1e-12, S
        assert np.abs(lse - ref_lse).max() <= 1e-12, S


def pin_mq_library_cross_check(o):
    p = custom("mqt", 2, 4, 2, 64, [50, 6], "f16", seed=15, tq=3)
    out, lse = o.attention_mq(p, 3)
    q = torch.from_numpy(_dec(p, p.q))
    k = torch.from_numpy(_dec(p, p.k))
    v = torch.from_numpy(_dec(p, p.v))
    for b, L in enumerate(p.lens):
        kk = k[int(p.cu[b]): int(p.cu[b + 1])]
        vv = v[int(p.cu[b]): int(p.cu[b + 1])]
        for t in range(3):
            mask = torch.arange(L) <= (L - 3 + t)
            for h in range(4):
                sc = (kk[:, h // 2, :] @ q[b, t, h]) * p.scale
                sc = sc.masked_fill(~mask, -math.inf)
                ref = torch.softmax(sc, 0) @ vv[:, h // 2, :]
                assert (out[b, t, h] - ref.numpy()).__abs__().max() <= 1e-12


def pin_mq_varsplit_merge_invariance(o):
    """Several tokens with per-sequence split counts merge back to the causal unsplit result
    (ragged batch with an empty sequence and sequences shorter than the token count, GQA,
    both layouts); S_b follows its closed form and the splits past S_b are empty."""
    for layout in (LAYOUT_VARLEN, LAYOUT_BHSD):
        lens = [300, 2, 0, 77, 1000]
        tq = 3
        p = custom("vsm", 5, 8, 2, 64, lens, "f16", layout=layout, seed=21, tq=tq,
                   kv_rows=1024 if layout == LAYOUT_BHSD else 0)
        ref, ref_lse = o.attention_mq(p, tq)
        for n, m in ((16, 64), (100, 4), (64, 1), (7, 200)):
            op, lp, sc = o.split_partials_var_mq(p, tq, n, m)
            out, lse = o.merge(op.reshape(-1, m, p.D), lp.reshape(-1, m))
            out = out.reshape(ref.shape)
            lse = lse.reshape(ref_lse.shape)
            assert np.abs(out - ref).max() <= 1e-12, (layout, n, m)
            fin = np.isfinite(ref_lse)
            assert np.array_equal(fin, np.isfinite(lse))
            assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12
            for b, L in enumerate(lens):
                assert sc[b] == (1 if L == 0 else min(m, -(-L // n)))
                assert np.isneginf(lp[b, :, :, sc[b]:]).all() and not op[b, :, :, sc[b]:].any()


def pin_mq_varsplit_uniform_counts(o):
    """When every sequence gets the same S_b = S, the per-sequence partials are the uniform
    ones of split_partials_mq, entry for entry (the same bounds floor(L*s/S))."""
    lens = [130, 150, 161, 145]
    tq = 4
    p = custom("vsu", 4, 6, 3, 64, lens, "bf16", seed=22, tq=tq)
    op, lp, sc = o.split_partials_var_mq(p, tq, 41, 8)      # ceil(L / 41) = 4 for every L here
    assert (sc == 4).all()
    ou, lu = o.split_partials_mq(p, tq, 4)
    assert np.array_equal(op[:, :, :, :4], ou) and np.array_equal(lp[:, :, :, :4], lu)
    assert np.isneginf(lp[:, :, :, 4:]).all()
    # tq = 1 is the single-token per-sequence function
    p1 = custom("vs1", 3, 8, 2, 64, [9, 100, 1], "f16", seed=23)
    a, la, sa = o.split_partials_var(p1, 16, 8)
    b, lb, sb = o.split_partials_var_mq(p1, 1, 16, 8)
    assert np.array_equal(a, b[:, 0]) and np.array_equal(la, lb[:, 0]) and np.array_equal(sa, sb)


ALL_PINS = [
    pin_f16_decoder, pin_bf16_decoder, pin_split_bounds_golden, pin_split_bounds_partition,
    pin_split_invariance, pin_weights_sum_to_one, pin_single_key, pin_single_key_lse,
    pin_constant_v, pin_gqa_packing, pin_hand_example, pin_q_zero_closed_form,
    pin_one_hot_dominance, pin_library_cross_check, pin_bhsd_matches_varlen,
    pin_empty_splits_and_sequences, pin_threads_deterministic, pin_rows_match_full,
    pin_rows_mq_match_full,
    pin_split_counts_golden, pin_varsplit_merge_invariance,
    pin_mq_causal_counts_golden, pin_mq_tq1_equals_single, pin_mq_token_equals_truncated_single,
    pin_mq_split_invariance, pin_mq_library_cross_check,
    pin_mq_varsplit_merge_invariance, pin_mq_varsplit_uniform_counts,
]
