"""The C-ABI library on the host: symbols, layout arithmetic, picker, argument checks.

Nothing here reaches a CUDA call: every case is rejected (or answered) by the
host-side code before any device work would be enqueued.
"""
import ctypes
import math
import os
import re

import pytest

import oracle
import split_kv_decode_decoding_gb300 as da

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "decode_attn_splitkv.h")


@pytest.fixture(scope="module")
def lib():
    da.build()
    return da.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(decode_attn_splitkv\w*)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) == 23
    assert sorted(names) == sorted(da.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        s = da.status_string(code)
        assert s and s != "unknown da_status"
    assert da.status_string(99) == "unknown da_status"


def test_device_timeout_status_and_layout_alias(lib):
    """The status the error readers return for a timed-out wait, and the varlen layout's
    second name, as the header declares them."""
    text = open(HEADER).read()
    assert re.search(r"DA_ERR_DEVICE_TIMEOUT\s*=\s*7", text)
    assert re.search(r"DA_LAYOUT_VARLEN_THD\s*=\s*DA_LAYOUT_VARLEN", text)
    assert da.DA_ERR_DEVICE_TIMEOUT == 7 and da.DA_LAYOUT_VARLEN_THD == da.DA_LAYOUT_VARLEN == 0
    assert da.status_string(da.DA_ERR_DEVICE_TIMEOUT).startswith("DA_ERR_DEVICE_TIMEOUT")
    v = ctypes.c_void_p
    assert lib.decode_attn_splitkv_noalloc_get_error(None, None) == da.DA_ERR_INVALID_ARG


def test_workspace_layout(lib):
    B, Hq, D, S = 3, 28, 128, 7
    lo = lib.decode_attn_splitkv_lse_offset()
    oo = lib.decode_attn_splitkv_opart_offset(B, Hq, S)
    assert lo == 256 and oo % 256 == 0 and oo >= lo + 4 * B * Hq * S
    assert da.workspace_size(B, Hq, D, S) == oo + 4 * B * Hq * S * D
    assert da.workspace_size(0, Hq, D, S) == 0
    assert da.workspace_size(B, Hq, D, 0) == 0
    assert da.workspace_size(B, Hq, D, da.DA_MAX_SPLITS + 1) == 0


def test_split_range_matches_oracle_bit_exact(lib):
    orc = oracle.default()
    for L in list(range(0, 300, 7)) + [4096, 8191, 131072, 2_000_000_000]:
        for S in (1, 2, 3, 4, 7, 16, 37, 152, 1000, 1024):
            for s in {0, 1, S // 2, S - 1}:
                if s < S:
                    assert da.split_range(L, S, s) == orc.split_range(L, S, s), (L, S, s)


@pytest.mark.parametrize("shape", [
    (2, 4, 1, 64, 37, 200), (8, 32, 32, 128, 4096, 4096), (64, 28, 4, 128, 512, 8192),
    (256, 16, 2, 128, 256, 256), (1, 16, 2, 128, 65536, 65536), (1, 16, 2, 128, 131072, 131072),
    (1, 32, 8, 128, 1024, 1024), (16, 32, 8, 128, 131072, 131072), (4, 64, 1, 128, 3, 9000),
])
def test_picker_properties(lib, shape):
    B, Hq, Hkv, D, mn, mx = shape
    for sm in (148, 152):
        S = da.num_splits(B, Hq, Hkv, D, mn, mx, sm)
        assert 1 <= S <= min(mn, da.DA_MAX_SPLITS)
        assert S == da.num_splits(B, Hq, Hkv, D, mn, mx, sm)
        cols = Hq // Hkv
        chunks = math.ceil(cols / (16 if cols > 8 else 8))   # 16-column items past 8 columns
        units = B * Hkv * chunks
        slots = sm * (2 if D == 128 else 4)
        if 2 * mn > mx:
            if 5 * units >= 4 * sm:
                # enough units for one wave: one split, or about 1.7 waves for a long stream
                kv_bytes = B * Hkv * mn * 4 * D
                assert S == (1 if kv_bytes <= 1.5e9 else max(1, round(1.68 * slots / units)))
            else:
                # about one item per SM, splits of at least 256 keys
                assert units * (S - 1) < sm
                assert S == 1 or mn // S >= 256
        else:
            # eight items per SM, or as many as keep the longest splits near two CTA shares
            # (16-column items: four per SM, four shares); a batch of at most 128
            # sequences none of which holds half the keys is handed out longest first:
            # six items per SM and four shares (16-column items: three and eight)
            wide = cols > 8
            total = mx + (B - 1) * mn
            sorted_ = B <= 128 and 2 * mx <= total
            per_sm = (3 if wide else 6) if sorted_ else (4 if wide else 8)
            shares = (8 if wide else 4) if sorted_ else (4 if wide else 2)
            share = total * Hkv * chunks / slots
            assert (units * (S - 1) < per_sm * sm or S == math.ceil(mx / (shares * share)))


def test_picker_choices_on_measured_workloads(lib):
    """Split counts the picker gives for shapes whose best split count was measured on a GB300."""
    sm = 152
    assert da.num_splits(16, 32, 8, 128, 8192, 8192, sm) == 1        # one wave of 128 items, no combine
    assert da.num_splits(16, 32, 8, 128, 32768, 32768, sm) == 4      # 2.1 GB stream: 512 items
    assert da.num_splits(16, 32, 8, 128, 131072, 131072, sm) == 4
    assert da.num_splits(8, 32, 32, 128, 4096, 4096, sm) == 1
    assert 16 <= da.num_splits(16, 32, 8, 128, 512, 131072, sm) <= 24   # one 128K sequence among 512s
    # Qwen heads (28 / 4), lengths 552 .. 8192, handed out longest first: S = 3 .. 8
    # measured 94.4, 93.8, 95.2, 96.6 us
    assert da.num_splits(64, 28, 4, 128, 552, 8192, sm) == 4
    # several query tokens: Hq passed as Hq * T_q
    assert da.num_splits(64, 28 * 2, 4, 128, 552, 8192, sm) == 2        # 14 columns: S 2..4: 99.7, 101.8, 103.4
    assert da.num_splits(64, 28 * 4, 4, 128, 552, 8192, sm) == 1        # 28 columns: S 1..3: 106.8, 114.2, 124.8
    # one 128K sequence among 512s with four tokens (16-column items): S 9: 153.0, 16: 113.7, 19: 114.7
    assert 16 <= da.num_splits(16, 32 * 4, 8, 128, 512, 131072, sm) <= 19


def test_picker_degenerate(lib):
    assert da.num_splits(2, 4, 1, 64, 0, 10, 152) == 1      # an empty sequence present
    assert da.num_splits(2, 4, 3, 64, 10, 10, 152) == 1     # Hq % Hkv != 0
    assert da.num_splits(2, 4, 1, 96, 10, 10, 152) == 1     # unsupported D
    assert da.num_splits(2, 4, 1, 64, 20, 10, 152) == 1     # min > max
    assert da.num_splits(1, 8, 1, 128, 1, 1, 152) == 1      # one key: one split


# --- argument checks (fake, aligned device addresses: never dereferenced) -------------
FAKE = 0x7f0000000000


def call_full(lib, **kw):
    a = dict(q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, cu=FAKE + 0x300000, B=2, Hq=4, Hkv=1,
             D=64, kv_rows=237, dt=0, lay=0, scale=0.125, S=4, out=FAKE + 0x400000,
             ws=FAKE + 0x500000, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    v = ctypes.c_void_p
    return lib.decode_attn_splitkv(v(a["q"]), v(a["k"]), v(a["v"]), v(a["cu"]), a["B"], a["Hq"],
                                   a["Hkv"], a["D"], a["kv_rows"], a["dt"], a["lay"], a["scale"],
                                   a["S"], v(a["out"]), v(a["ws"]), a["ws_bytes"], v(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), da.DA_ERR_INVALID_ARG),
    (dict(Hq=0), da.DA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), da.DA_ERR_INVALID_ARG),
    (dict(kv_rows=-1), da.DA_ERR_INVALID_ARG),
    (dict(S=0), da.DA_ERR_INVALID_ARG),
    (dict(S=da.DA_MAX_SPLITS + 1), da.DA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), da.DA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), da.DA_ERR_INVALID_ARG),
    (dict(dt=2), da.DA_ERR_INVALID_ARG),
    (dict(lay=2), da.DA_ERR_INVALID_ARG),
    (dict(D=96), da.DA_ERR_UNSUPPORTED),
    (dict(D=256), da.DA_ERR_UNSUPPORTED),
    (dict(q=0), da.DA_ERR_INVALID_ARG),
    (dict(cu=0), da.DA_ERR_INVALID_ARG),
    (dict(ws=0), da.DA_ERR_INVALID_ARG),
    (dict(k=0), da.DA_ERR_INVALID_ARG),
    (dict(out=0), da.DA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), da.DA_ERR_ALIGNMENT),
    (dict(k=FAKE + 0x100004), da.DA_ERR_ALIGNMENT),
    (dict(cu=FAKE + 0x300002), da.DA_ERR_ALIGNMENT),
    (dict(ws=FAKE + 0x500080), da.DA_ERR_ALIGNMENT),
    (dict(out=FAKE + 0x400008), da.DA_ERR_ALIGNMENT),
    (dict(ws_bytes=1000), da.DA_ERR_WORKSPACE_TOO_SMALL),
])
def test_host_checks(lib, kw, code):
    assert call_full(lib, **kw) == code


def test_other_entry_points_reject_bad_args(lib):
    v = ctypes.c_void_p
    bits = ctypes.c_uint32()
    assert lib.decode_attn_splitkv_get_error(None, ctypes.byref(bits), None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_get_error(v(FAKE + 64), ctypes.byref(bits), None) == da.DA_ERR_ALIGNMENT
    assert lib.decode_attn_splitkv_workspace_init(None, 1 << 20, None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_workspace_init(v(FAKE), 100, None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_selftest_timeout(v(FAKE), 1 << 20, 0, None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_combine(2, 4, 64, 4, 0, None, v(FAKE), 1 << 20, None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_combine(2, 4, 96, 4, 0, v(FAKE), v(FAKE), 1 << 20, None) == da.DA_ERR_UNSUPPORTED
    assert lib.decode_attn_splitkv_combine(2, 4, 64, 4, 0, v(FAKE), v(FAKE), 100, None) == da.DA_ERR_WORKSPACE_TOO_SMALL
    assert lib.decode_attn_splitkv_partial(v(FAKE), v(FAKE), v(FAKE), v(FAKE), 2, 4, 1, 64, 237, 0, 0,
                                           0.125, 4, v(FAKE), 10, None) == da.DA_ERR_WORKSPACE_TOO_SMALL


def test_binding_refuses_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("split_kv_decode_decoding_gb300")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError):
            mod.load(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def test_varsplit_plan(lib):
    n, m = da.varsplit_plan(64, 28, 4, 128, 64 * 4352, 8192, 152)
    assert n % 64 == 0 and n >= 256 and m == -(-8192 // n)
    # items of about 0.4 of one CTA's share (304 CTAs at head_dim 128): 2.5 per CTA
    items = 64 * 4352 * 4 / n
    assert 2.5 * 304 * 0.9 <= items <= 2.5 * 304 * 1.05
    # four query tokens: 28 columns per KV head take two chunks, each a pass over the keys
    n4, m4 = da.varsplit_plan(64, 28 * 4, 4, 128, 64 * 4352, 8192, 152)
    assert 2 * 64 * 4352 * 4 / n4 <= 2.5 * 304 * 1.05 and n4 >= 2 * n - 64 and m4 == -(-8192 // n4)
    # one long sequence among short ones: it gets at most about half the CTAs' worth of items
    n, m = da.varsplit_plan(16, 32, 8, 128, 131072 + 15 * 512, 131072, 152)
    assert n % 64 == 0 and 8 * m <= 304 // 2 + 8 and n >= 2 * 131072 * 8 // 304
    n, m = da.varsplit_plan(2, 4, 1, 64, 237, 200, 152)
    assert (n, m) == (256, 1)
    with pytest.raises(ValueError):
        da.varsplit_plan(2, 4, 3, 64, 237, 200, 152)


def test_varsplit_host_checks(lib):
    v = ctypes.c_void_p
    args = lambda **kw: [v(kw.get("q", FAKE)), v(FAKE + 0x100000), v(FAKE + 0x200000), v(FAKE + 0x300000),
                         kw.get("B", 2), 4, 1, 64, 237, 0, 0, 0.125, kw.get("n", 64), kw.get("m", 4),
                         v(FAKE + 0x400000), v(FAKE + 0x500000), 1 << 20, None]
    assert lib.decode_attn_splitkv_varsplit(*args(n=0)) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_varsplit(*args(m=0)) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_varsplit(*args(m=da.DA_MAX_SPLITS + 1)) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_splitkv_varsplit(*args(B=da.DA_MAX_VARSPLIT_BATCH + 1)) == da.DA_ERR_UNSUPPORTED
    assert lib.decode_attn_splitkv_varsplit(*args(q=FAKE + 2)) == da.DA_ERR_ALIGNMENT


def test_multiquery_host_checks(lib):
    v = ctypes.c_void_p

    def call(T=2, S=4, ws_bytes=1 << 20, q=FAKE):
        return lib.decode_attn_splitkv_multiquery(v(q), v(FAKE + 0x100000), v(FAKE + 0x200000),
                                                  v(FAKE + 0x300000), 2, T, 4, 1, 64, 237, 0, 0, 0.125,
                                                  S, v(FAKE + 0x400000), v(FAKE + 0x500000), ws_bytes,
                                                  None)
    assert call(T=0) == da.DA_ERR_INVALID_ARG
    assert call(T=da.DA_MAX_QUERY_TOKENS + 1) == da.DA_ERR_INVALID_ARG
    assert call(S=0) == da.DA_ERR_INVALID_ARG
    assert call(q=FAKE + 4) == da.DA_ERR_ALIGNMENT
    need = da.workspace_size(2 * 2, 4, 64, 4)
    assert call(ws_bytes=need - 1) == da.DA_ERR_WORKSPACE_TOO_SMALL


def test_multiquery_varsplit_host_checks(lib):
    v = ctypes.c_void_p

    def call(T=2, n=64, m=4, B=2, ws_bytes=1 << 20, q=FAKE):
        return lib.decode_attn_splitkv_multiquery_varsplit(v(q), v(FAKE + 0x100000), v(FAKE + 0x200000),
                                                           v(FAKE + 0x300000), B, T, 4, 1, 64, 237, 0, 0,
                                                           0.125, n, m, v(FAKE + 0x400000), v(FAKE + 0x500000),
                                                           ws_bytes, None)
    assert call(n=0) == da.DA_ERR_INVALID_ARG
    assert call(m=0) == da.DA_ERR_INVALID_ARG
    assert call(m=da.DA_MAX_SPLITS + 1) == da.DA_ERR_INVALID_ARG
    assert call(T=0) == da.DA_ERR_INVALID_ARG
    assert call(T=da.DA_MAX_QUERY_TOKENS + 1) == da.DA_ERR_INVALID_ARG
    assert call(B=da.DA_MAX_VARSPLIT_BATCH + 1, ws_bytes=1 << 30) == da.DA_ERR_UNSUPPORTED
    assert call(q=FAKE + 4) == da.DA_ERR_ALIGNMENT
    need = da.workspace_size(2 * 2, 4, 64, 4)
    assert call(ws_bytes=need - 1) == da.DA_ERR_WORKSPACE_TOO_SMALL


def test_multiquery_tmem_host_checks(lib):
    """The tcgen05 arm takes G * T_q > 8 with G <= 32 only; the checks launch nothing."""
    v = ctypes.c_void_p

    def call(T=4, Hq=8, Hkv=2, S=2, ws_bytes=1 << 22):
        return lib.decode_attn_splitkv_multiquery_tmem(v(FAKE), v(FAKE + 0x100000), v(FAKE + 0x200000),
                                                       v(FAKE + 0x300000), 2, T, Hq, Hkv, 64, 237, 0, 0,
                                                       0.125, S, v(FAKE + 0x400000), v(FAKE + 0x500000),
                                                       ws_bytes, None)
    assert call(T=2) == da.DA_ERR_UNSUPPORTED              # G * T_q = 8: one n-tile, not this arm
    assert call(T=1, Hq=66, Hkv=1) == da.DA_ERR_UNSUPPORTED   # G = 66 > 32
    assert call(T=0) == da.DA_ERR_INVALID_ARG
    assert call(S=0) == da.DA_ERR_INVALID_ARG
    need = da.workspace_size(2 * 4, 8, 64, 2)
    assert call(ws_bytes=need - 1) == da.DA_ERR_WORKSPACE_TOO_SMALL


def test_time_model_formula_by_hand(lib):
    """One sequence, one KV head, D = 128, explicit parameters: the formula worked by hand.

    L = 1000, S = 2: splits of 500 keys, rounded up to 512 (16-key boxes), 4*128 = 512 B
    per key -> 262144 B each. With t0 = 5, t_item = 1, r_cta = 65536 B/us, bw = 1e6,
    t_comb = 2, bw_comb = 1e6, kappa = 0.5: two items on two free CTAs; each CTA waits
    t_item = 1 us, then the two stream together at min(65536, 1e6 / 2) = 65536 B/us for
    4 us, so the makespan is 5 us. The last-item term is 0.5 * 262144 / (1e6 / 2) =
    0.262144 us; workspace 1*1*1*2*129*4 = 1032 B. T = 5 + 5 + 0.262144 + 2 + 0.001032.
    """
    params = [5.0, 1.0, 65536.0, 1e6, 2.0, 1e6, 0.5, 32768.0]
    t = da.model_us([1000], 1, 1, 128, 2, 152, params=params)
    assert abs(t - (5 + 5 + 0.262144 + 2 + 0.001032)) < 1e-9
    # one split: no combine term, one 1008-key item (1000 rounded up): 1 + 1008*512/65536,
    # last-item term 0.5 * 516096 / 1e6
    t1 = da.model_us([1000], 1, 1, 128, 1, 152, params=params)
    assert abs(t1 - (5 + 1 + 1008 * 512 / 65536 + 0.5 * 516096 / 1e6)) < 1e-9
    # bandwidth-bound: four items streaming together share bw = 1e5 B/us (25000 each,
    # below r_cta): 1 + 262144 / 25000 us; last-item term 0.5 * 262144 / 25000; the
    # combine reads 2*1*2*129*4 = 2064 B
    params_bw = [5.0, 1.0, 65536.0, 1e5, 2.0, 1e6, 0.5, 32768.0]
    t4 = da.model_us([1000, 1000], 1, 1, 128, 2, 152, params=params_bw)
    assert abs(t4 - (5 + 1 + 262144 / 25000 + 0.5 * 262144 / 25000 + 2 + 0.002064)) < 1e-9


def test_time_model_per_sequence_by_hand(lib):
    """Per-sequence counts, worked by hand: lengths [1000, 300], split_len 500, max_splits 4.

    S_b = 2 and 1: two items of 500 keys (512 after rounding: 262144 B) and one of 300 (304:
    155648 B), in sequence order, three CTAs streaming at min(65536, 1e6 / 3) = 65536 B/us
    after t_item = 1 us: the makespan is 1 + 262144 / 65536 = 5 us. Last-item term
    0.5 * 262144 / (1e6 / 3); the combine reads the two split rows of sequence 0 only:
    2 * 129 * 4 = 1032 B."""
    params = [5.0, 1.0, 65536.0, 1e6, 2.0, 1e6, 0.5, 32768.0]
    t = da.model_varsplit_us([1000, 300], 1, 1, 128, 500, 4, 152, params=params)
    assert abs(t - (5 + 5 + 0.5 * 262144 / (1e6 / 3) + 2 + 0.001032)) < 1e-9
    # every sequence in one split: the uniform model with S = 1 (same order here)
    assert abs(da.model_varsplit_us([1000, 300], 1, 1, 128, 2000, 1, 152, params=params)
               - da.model_us([1000, 300], 1, 1, 128, 1, 152, params=params)) < 1e-12
    assert da.model_varsplit_us([1000, 300], 1, 1, 128, 0, 4, 152) < 0       # split_len < 1


def test_time_model_queue_order(lib):
    """With uniform splits the model hands out a batch of up to 128 sequences longest first, as
    the split step does: the order of the lengths does not matter. Per-sequence counts go out in
    sequence order, where a long sequence at the end of the queue costs more."""
    lens = [512] * 30 + [65536]
    rev = [65536] + [512] * 30
    t_end = da.model_us(lens, 32, 8, 128, 4, 152)
    t_start = da.model_us(rev, 32, 8, 128, 4, 152)
    assert abs(t_end - t_start) < 1e-9
    # 16 splits of the long sequence x 8 KV heads + 240 short items: more items than the 304 CTAs
    v_end = da.model_varsplit_us(lens, 32, 8, 128, 4096, 16, 152)
    v_start = da.model_varsplit_us(rev, 32, 8, 128, 4096, 16, 152)
    assert v_end > v_start


def test_time_model_properties(lib):
    base = da.model_us([4096] * 8, 32, 32, 128, 1, 152)
    assert base > 0
    assert da.model_us([8192] * 8, 32, 32, 128, 1, 152) > 1.5 * base   # twice the bytes
    # one long sequence: splitting it helps a lot
    assert da.model_us([131072], 16, 2, 128, 64, 152) < 0.2 * da.model_us([131072], 16, 2, 128, 1, 152)
    S, t = da.model_best_splits([131072], 16, 2, 128, 152)
    assert 8 <= S <= 256 and t > 0
    assert da.model_us([100], 4, 3, 128, 1, 152) < 0          # Hq % Hkv != 0
    assert da.model_best_splits([5, 3], 4, 1, 128, 152)[0] <= 3


def call_noalloc(lib, **kw):
    a = dict(q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, cu=FAKE + 0x300000, B=2, Hq=4, Hkv=1,
             D=64, kv_rows=237, dt=0, lay=0, scale=0.125, S=4, out=FAKE + 0x400000, stream=None)
    a.update(kw)
    v = ctypes.c_void_p
    return lib.decode_attn_splitkv_noalloc(v(a["q"]), v(a["k"]), v(a["v"]), v(a["cu"]), a["B"], a["Hq"],
                                           a["Hkv"], a["D"], a["kv_rows"], a["dt"], a["lay"], a["scale"],
                                           a["S"], v(a["out"]), v(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(B=64, Hq=28, Hkv=4, D=128, S=16), da.DA_ERR_SCRATCH_LIMIT),   # 14.9 MB of scratch
    (dict(B=4096, Hq=64, Hkv=8, D=128, S=1), da.DA_ERR_SCRATCH_LIMIT),
    (dict(B=0), da.DA_ERR_INVALID_ARG),
    (dict(S=0), da.DA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), da.DA_ERR_INVALID_ARG),
    (dict(D=96), da.DA_ERR_UNSUPPORTED),
    (dict(q=0), da.DA_ERR_INVALID_ARG),
    (dict(out=0), da.DA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), da.DA_ERR_ALIGNMENT),
    (dict(cu=FAKE + 0x300002), da.DA_ERR_ALIGNMENT),
    (dict(out=FAKE + 0x400008), da.DA_ERR_ALIGNMENT),
])
def test_noalloc_host_checks(lib, kw, code):
    """The no-allocation entry point refuses bad arguments on the host, before it looks up
    its scratch array on a device (there is none here: a lookup would fail with DA_ERR_CUDA)."""
    assert call_noalloc(lib, **kw) == code
