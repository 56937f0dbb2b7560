"""bench.py on the GPU: the JSON line carries every field of its contract, with sane values."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_default_line_has_the_contract_fields():
    d = bench_line("--steps", "20", "--warmup", "3", "--e2e-steps", "3")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "cpu_baseline", "back_to_back"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    # the largest single-GPU workload: Llama-3.1-8B heads, 16 sequences of 131072 keys, bf16
    assert d["config"]["workload"] == "llama_S131072_B16" and "flush" in d["config"]["l2"]
    assert d["dtype"] == "bf16"
    assert 1000.0 < d["value"] < 12000.0                       # KV GB/s on one GB300
    assert abs(d["pct_of_nominal_8tbs"] - 100.0 * d["value"] / 8000.0) < 0.01
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3 and 0.1 < r["frac"] < 1.5
    kv = 2 * 16 * 8 * 131072 * 128 * 2
    assert r["alg_bytes_per_launch"] >= kv                     # at least the K/V bytes
    if r["traffic"] is not None:                                # recorded for this kernel source
        assert 0.9 * r["alg_bytes_per_launch"] < r["traffic"] < 1.2 * r["alg_bytes_per_launch"]
    e = d["e2e"]
    assert e["unit"] == "GB/s" and 0 < e["value"] < d["value"]
    assert e["h2d_bytes_per_step"] >= kv and e["d2h_bytes_per_step"] == 16 * 32 * 128 * 2
    assert d["gpu_launches"] > 0
    # NVML samples every 2 ms: even a short timed region has clock samples
    k = d["clocks"]
    assert k["source"] == "nvml" and k["samples"] >= 3 and k["sm_mhz"] > 0 and k["sm_max_mhz"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["one_thread"]["value"] > 0
    assert d["back_to_back"]["inputs_exceed_l2"] is True and d["back_to_back"]["value"] > 0


def test_multi_token_and_comparison_arms_run():
    mq = bench_line("--workload", "qwen_varlen", "--tq", "2", "--steps", "10", "--warmup", "3", "--e2e-steps", "2",
                    "--no-cpu-baseline", "--no-clocks")
    assert mq["config"]["query_tokens"] == 2 and mq["value"] > 0 and mq["e2e"]["value"] > 0
    tm = bench_line("--workload", "qwen_varlen", "--tq", "4", "--tmem-math", "--steps", "10", "--warmup", "3",
                    "--no-cpu-baseline", "--no-clocks")
    assert "tcgen05" in tm["config"]["products"] and tm["value"] > 0 and tm["roofline"]["traffic"] is None
    cc = bench_line("--workload", "codellama_B64_S1024", "--cuda-core-math", "--steps", "10", "--warmup", "3",
                    "--no-cpu-baseline", "--no-clocks")
    assert "CUDA-core" in cc["config"]["products"] and cc["value"] > 0
