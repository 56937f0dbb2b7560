"""The seeded input generator: determinism, counter addressing, rounding, distribution."""
import math

import numpy as np

import synth
from synth.workloads import all_workload_names, workload


def test_counter_addressing_and_determinism():
    a = synth.normal_bits(0, 2, 300_000, "f16")
    b = synth.normal_bits(0, 2, 300_000, "f16")
    assert np.array_equal(a, b)
    tail = synth.normal_bits(0, 2, 1000, "f16", first=123_456)
    assert np.array_equal(tail, a[123_456:124_456])
    other = synth.normal_bits(0, 3, 1000, "f16")
    assert not np.array_equal(other, a[:1000])
    assert not np.array_equal(synth.normal_bits(1, 2, 1000, "f16"), a[:1000])


def test_f16_rounding_matches_numpy():
    x = synth.normal_f64(5, 9, 200_000) * np.float64(3.0)
    x = np.concatenate([x, [65504.0, 65519.99, 65520.0, 1e-8, -3e-5, 2.0 ** -25, 0.0, -0.0]])
    got = np.array([synth.round_f16(v) for v in x], dtype=np.uint16)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def _bf16_rne(x: float) -> int:
    """Exact double -> bfloat16 rounding with Python's round-half-even on exact doubles."""
    if x == 0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if a < 2.0 ** -126:
        q = round(a * 2.0 ** 133)
        return sign | q
    m, e = math.frexp(a)
    r = round(math.ldexp(a, 8 - e))
    E = e - 1
    if r == 256:
        r, E = 128, E + 1
    return sign | ((E + 127) << 7) | (r - 128)


def test_bf16_rounding_exact():
    x = synth.normal_f64(6, 9, 50_000) * np.float64(7.0)
    x = np.concatenate([x, [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3e-39, -1e-40]])
    for v in x:
        assert synth.round_bf16(v) == _bf16_rne(float(v)), v


def test_normal_moments():
    z = synth.normal_f64(0, 1, 1_000_000)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert 0.30 < np.mean(np.abs(z) > 1.0) < 0.335


def test_uniform_int_range():
    u = synth.uniform_int(0, 4, 100_000, 512, 8192)
    assert u.min() >= 512 and u.max() <= 8192
    assert abs(u.mean() - (512 + 8192) / 2) < 40


def test_workload_shapes():
    names = all_workload_names()
    assert len(names) == 3 + 10 + 8
    p = workload("tiny")
    assert p.q.shape == (2, 4, 64) and p.k.shape == (237, 1, 64)
    assert list(p.cu) == [0, 37, 237] and p.num_splits == 4
    assert p.kv_bytes == 2 * 237 * 64 * 2
    q = workload("qwen_varlen", data=False)
    assert q.B == 64 and q.Hq == 28 and q.Hkv == 4 and min(q.lens) >= 512 and max(q.lens) <= 8192
    m = workload("mha_bhsd", data=False)
    assert m.kv_bytes == 536_870_912
    c = workload("codellama_B1_S131072", data=False)
    assert c.kv_bytes == 134_217_728
    ll = workload("llama_S131072_B16", data=False)
    assert ll.kv_bytes == 8_589_934_592 and ll.dtype == "bf16"
