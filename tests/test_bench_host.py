"""Host-side pieces of bench.py: rank aggregation (2 gloo ranks on CPU), clock parsing."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks(3.5) == 3.5


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.kind = "nvidia-smi"
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    c.lines = []
    assert c.summary()["reasons"] == ["no samples"]


def test_nvml_clock_summary_parsing():
    """The NVML child prints 'sm_mhz,max_mhz,reason bits'; bit 0x4 is the software power cap,
    0x8 the hardware slowdown (nvml.h clock-event reasons); idle (0x1) is not a slowdown."""
    c = bench.ClockSampler(0)
    c.kind = "nvml"
    c.lines = ["2070,2070,0", "1995,2070,4", "2070,2070,1", "1500,2070,12"]
    s = c.summary()
    assert s["samples"] == 4 and s["sm_mhz"] == 2032.5 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"] and s["source"] == "nvml"


def test_clock_sampler_without_a_gpu_returns_no_samples_or_a_summary():
    """Here (no GPU, no NVML) the child reports it is unavailable and the sampler falls back;
    whatever it gets, it never raises and never blocks."""
    with bench.ClockSampler(0, interval_ms=1.0) as c:
        pass
    s = c.summary()
    assert "reasons" in s


def test_recorded_traffic_needs_current_kernel(tmp_path, monkeypatch):
    f = tmp_path / "t.json"
    f.write_text('{"entries": [{"kernel_sha": "%s", "workload": "w", "num_splits": 3, '
                 '"dram_bytes_per_launch": 123.0}]}' % bench.kernel_sha())
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w", 3)[0] == 123.0
    assert bench.recorded_traffic("w", 4) == (None, None)
    f.write_text('{"entries": [{"kernel_sha": "old", "workload": "w", "num_splits": 3, '
                 '"dram_bytes_per_launch": 1.0}]}')
    assert bench.recorded_traffic("w", 3) == (None, None)
    # a capture on a smaller case stands for a larger one of the same shape, scaled
    f.write_text('{"entries": [{"kernel_sha": "%s", "workload": "small", "num_splits": 4, '
                 '"dram_bytes_per_launch": 100.0, "scale_to": {"big": 4.0}}]}' % bench.kernel_sha())
    b, src = bench.recorded_traffic("big", 4)
    assert b == 400.0 and "small" in src and "x4.0" in src
    assert bench.recorded_traffic("big", 3) == (None, None)
    assert bench.recorded_traffic("small", 4)[0] == 100.0


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference times the float64 oracle and prints the contract's line."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"
