"""Benchmark: split-KV decode attention on one GB300 (or N replicas under torchrun).

Prints ONE JSON line (rank 0). A step is one decode_attn_splitkv call over the
whole workload (the split kernel then the combine kernel, chained by programmatic
dependent launch), timed with CUDA events on its stream. After the K steps,
K/2 more steps call decode_attn_splitkv_partial and decode_attn_splitkv_combine
(the same two launches) with events around the split kernel alone, for its roofline. L2 is flushed between steps by writing a buffer twice its size, then reading another.

  value      KV-read GB/s = 2 * sum(L_b) * Hkv * D * 2 bytes / mean step time
  e2e        the same metric through decode_attn_splitkv with the inputs copied
             host->device (pinned) and the output copied back inside each step
  roofline   the split kernel: algorithmic bytes per launch / its mean event time,
             against the measured HBM copy bandwidth
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample

--impl reference times the float64 CPU oracle alone (there is no other
implementation of this method to run) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/call and KV-read HBM GB/s (% of GB300 peak)"
DEFAULT_WORKLOAD = "llama_S131072_B16"
# the sources the library's own kernels are compiled from (recorded ncu traffic is current only
# while these are unchanged)
CU_SRCS = [os.path.join(ROOT, "split_kv_decode_decoding_gb300", "csrc", n)
           for n in ("decode_attn_splitkv.cu", "split_common.cuh", "geometry.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=0, help="override the split-count picker")
    ap.add_argument("--varsplit", action="store_true",
                    help="per-sequence split counts (decode_attn_splitkv_varsplit, or "
                         "decode_attn_splitkv_multiquery_varsplit with --tq > 1) with its planner")
    ap.add_argument("--split-len", type=int, default=0, help="override the planner's split_len")
    ap.add_argument("--cuda-core-math", action="store_true",
                    help="time the split step with its products on CUDA-core fp32 FMAs instead of "
                         "tensor cores (the comparison arm; uniform splits, one query token, G <= 8)")
    ap.add_argument("--tmem-math", action="store_true",
                    help="run the tcgen05 / tensor-memory comparison arm (G * T_q > 8, G <= 32)")
    ap.add_argument("--fa2-style", action="store_true",
                    help="comparison: no split and one query head per unit (K/V repeated per "
                         "query head, as FlashAttention-style decode reads them); GB/s still "
                         "counts the GQA cache bytes")
    ap.add_argument("--tq", type=int, default=1,
                    help="query tokens per sequence (decode_attn_splitkv_multiquery when > 1)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--e2e-buffers", type=int, default=2,
                    help="device input sets the end-to-end steps alternate (2: a step's copies overlap "
                         "the previous step's call)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams the e2e leg spreads its host->device K/V copies over")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="do not flush L2 between steps")
    ap.add_argument("--read-probe", default="",
                    help="instead of the decode call, time the read-ceiling probe (a bare bulk-copy "
                         "stream through shared memory) over these buffer sizes in bytes, comma "
                         "separated, with the same flush and event pair; prints one JSON line")
    ap.add_argument("--probe-ctas-per-sm", type=int, default=2)
    ap.add_argument("--probe-chunk", type=int, default=16384)
    ap.add_argument("--probe-stages", type=int, default=4)
    ap.add_argument("--clock-sampler", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--clock-interval-ms", type=float, default=2.0, help=argparse.SUPPRESS)
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of a per-rank float over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for path in CU_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, S: int):
    """DRAM bytes per split-kernel launch from a committed ncu capture, if it is current:
    (bytes, source). An entry captured on a smaller case may name larger workloads of the
    same shape and split count in "scale_to" with the factor of units (keys) they process."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, None
    sha = kernel_sha()
    for e in d.get("entries", []):
        if e.get("kernel_sha") == sha and e.get("workload") == workload and e.get("num_splits") == S:
            return float(e["dram_bytes_per_launch"]), "ncu capture of this workload"
    for e in d.get("entries", []):
        f = e.get("scale_to", {}).get(workload)
        if e.get("kernel_sha") == sha and e.get("num_splits") == S and f:
            return (float(e["dram_bytes_per_launch"]) * float(f),
                    f"ncu capture of {e['workload']} scaled x{f} by the keys processed")
    return None, None


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*): read-only sampling
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def nvml_sampler_main(index: int, interval_ms: float) -> int:
    """Child process: print 'sm_mhz,max_mhz,reasons' every interval_ms until stdin closes.

    Reads the SM clock, its maximum and the clock-event reasons through NVML
    (libnvidia-ml, read-only queries); prints 'ready' once the first sample is taken."""
    import ctypes
    import select
    try:
        nv = ctypes.CDLL("libnvidia-ml.so.1")
    except OSError:
        print("unavailable", flush=True)
        return 0
    if nv.nvmlInit_v2() != 0:
        print("unavailable", flush=True)
        return 0
    h = ctypes.c_void_p()
    if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
        print("unavailable", flush=True)
        return 0
    reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
        getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
    clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
    first = True
    while True:
        ok = (nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and      # NVML_CLOCK_SM
              nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
              reasons_fn(h, ctypes.byref(rs)) == 0)
        if ok:
            print(f"{clk.value},{mx.value},{rs.value}", flush=True)
        if first:
            print("ready", flush=True)
            first = False
        r, _, _ = select.select([sys.stdin], [], [], interval_ms / 1000.0)
        if r and not sys.stdin.readline():
            break
    nv.nvmlShutdown()
    return 0


class ClockSampler:
    """SM clock and clock-event reasons sampled every 2 ms while the timed region runs, by a
    child process through NVML (the region of one bench run can be tens of milliseconds, too
    short for nvidia-smi's loop); nvidia-smi's 100 ms loop when NVML cannot be loaded."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: float = 2.0):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.kind = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                [sys.executable, os.path.abspath(__file__), "--clock-sampler", str(self.index),
                 "--clock-interval-ms", str(self.interval_ms)],
                stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            head = []
            while True:
                ln = self.proc.stdout.readline()
                if not ln or ln.strip() in ("ready", "unavailable"):
                    break
                head.append(ln)
            if ln.strip() == "ready":
                self.kind = "nvml"
                self.lines = head
                return self
            self.proc.wait(timeout=5)
        except (OSError, subprocess.TimeoutExpired):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.kind = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            try:
                if self.kind == "nvml":
                    out, _ = self.proc.communicate(input="", timeout=10)
                else:
                    self.proc.terminate()
                    out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines += [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                if self.kind == "nvml" and len(f) == 3:
                    sm.append(float(f[0]))
                    smax.append(float(f[1]))
                    bits = int(f[2])
                    reasons.update(n for b, n in NVML_REASONS.items() if bits & b)
                elif self.kind == "nvidia-smi" and len(f) >= 9:
                    sm.append(float(f[1]))
                    smax.append(float(f[2]))
                    reasons.update(n for n, v in zip(names, f[5:9]) if v.lower() == "active")
            except ValueError:
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": self.kind}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "source": self.kind,
                "interval_ms": self.interval_ms if self.kind == "nvml" else 100}


def problem_tensors(p, device):
    import numpy as np
    import torch
    dt = torch.float16 if p.dtype == "f16" else torch.bfloat16

    def host(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt)

    return host(p.q), host(p.k), host(p.v), torch.from_numpy(p.cu.astype(np.int32))


def cpu_oracle_sample(p, budget_s: float = 12.0, steps=None):
    """Time the float64 oracle on (b, h) rows of the workload: returns (GB/s, cores, desc, per-step s)."""
    import numpy as np

    import oracle
    orc = oracle.default()
    cores = os.cpu_count() or 1
    rows_b = np.repeat(np.arange(p.B), p.Hq).astype(np.int32)
    rows_h = np.tile(np.arange(p.Hq), p.B).astype(np.int32)
    nrows = rows_b.size
    # probe one row per thread to size the sample
    probe = min(nrows, cores)
    t0 = time.perf_counter()
    orc.attention_rows(p, rows_b[:probe], rows_h[:probe], nthreads=cores)
    t_probe = max(time.perf_counter() - t0, 1e-6)
    per_row = t_probe / probe * cores          # CPU-seconds per row
    if steps is None:
        want = int(budget_s * cores / per_row)
        n = max(probe, min(nrows, want))
        reps = max(1, min(20, want // nrows)) if n == nrows else 1
        sel = np.linspace(0, nrows - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        for _ in range(reps):
            orc.attention_rows(p, rows_b[sel], rows_h[sel], nthreads=cores)
        dt = time.perf_counter() - t0
        frac = n * reps / nrows
        gbs = p.kv_bytes * frac / dt / 1e9
        desc = (f"{n} of {nrows} (b, h) rows of {p.name} (full key ranges) x {reps} passes, "
                f"float64, {cores} threads, {dt:.2f} s wall")
        return gbs, cores, desc, dt
    budget_per_step = budget_s / steps
    n = max(1, min(nrows, int(budget_per_step * cores / per_row)))
    return n, nrows, cores


def cpu_oracle_one_thread(p, budget_s: float = 4.0):
    """The float64 oracle on one thread over (b, h) rows of the workload: returns (GB/s, desc)."""
    import numpy as np

    import oracle
    orc = oracle.default()
    rows_b = np.repeat(np.arange(p.B), p.Hq).astype(np.int32)
    rows_h = np.tile(np.arange(p.Hq), p.B).astype(np.int32)
    nrows = rows_b.size
    t0 = time.perf_counter()
    orc.attention_rows(p, rows_b[:1], rows_h[:1], nthreads=1)
    per_row = max(time.perf_counter() - t0, 1e-6)
    n = max(1, min(nrows, int(budget_s / per_row)))
    sel = np.linspace(0, nrows - 1, n).astype(np.int64)
    t0 = time.perf_counter()
    orc.attention_rows(p, rows_b[sel], rows_h[sel], nthreads=1)
    dt = time.perf_counter() - t0
    gbs = p.kv_bytes * (n / nrows) / dt / 1e9
    return gbs, f"{n} of {nrows} (b, h) rows, float64, 1 thread, {dt:.2f} s wall"


def run_reference(args, p, ws_, rank):
    """--impl reference: the float64 oracle alone, each step a bounded sample of rows."""
    import numpy as np

    import oracle
    if rank != 0:
        return None
    orc = oracle.default()
    n, nrows, cores = cpu_oracle_sample(p, budget_s=150.0, steps=args.steps + args.warmup)
    rows_b = np.repeat(np.arange(p.B), p.Hq).astype(np.int32)
    rows_h = np.tile(np.arange(p.Hq), p.B).astype(np.int32)
    times = []
    for i in range(args.warmup + args.steps):
        sel = (np.arange(n) * (nrows // n) + i) % nrows
        t0 = time.perf_counter()
        orc.attention_rows(p, rows_b[sel], rows_h[sel], nthreads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    frac = n / nrows
    step = sum(times) / len(times)
    value = p.kv_bytes * frac / step / 1e9
    sample = (f"{n} of {nrows} (b, h) rows per step of {p.name}, float64 oracle, {cores} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, None),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def workload_config(p, S):
    return {"workload": p.name, "batch": p.B, "q_heads": p.Hq, "kv_heads": p.Hkv,
            "head_dim": p.D, "kv_lens": (p.lens[0] if len(set(p.lens)) == 1 else
                                         f"{min(p.lens)}..{max(p.lens)} (mean {sum(p.lens) / len(p.lens):.0f})"),
            "layout": "bhsd" if p.layout == 1 else "varlen", "in_dtype": p.dtype,
            "query_tokens": p.tq,
            "num_splits": S, "kv_bytes": p.kv_bytes,
            "l2": "flushed between steps (write then read of 2x L2 size)"
                  + ("; the K/V inputs also exceed L2" if p.kv_bytes > 129e6 else "")}


def run_read_probe(args):
    """Time the read-ceiling probe over buffers of the given sizes: L2 flushed before each
    launch exactly as for the decode call, CUDA events around the launch alone."""
    import ctypes

    import torch

    from split_kv_decode_decoding_gb300.build import build_probe
    lib = ctypes.CDLL(build_probe())
    lib.read_probe.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_void_p, ctypes.c_void_p]
    lib.read_probe.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = []
    for nbytes in [int(x) for x in args.read_probe.split(",") if x]:
        nbytes -= nbytes % 16
        buf = torch.ones(nbytes // 2, dtype=torch.float16, device=dev)
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush_w.fill_(1)
                flush_r.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                rc = lib.read_probe(ctypes.c_void_p(buf.data_ptr()), nbytes, args.probe_ctas_per_sm,
                                    args.probe_chunk, args.probe_stages, ctypes.c_void_p(err.data_ptr()),
                                    ctypes.c_void_p(stream.cuda_stream))
                if rc != 0:
                    raise RuntimeError(f"read_probe returned {rc}")
                e1.record(stream)
                if i >= args.warmup:
                    times.append((e0, e1))
            torch.cuda.synchronize(dev)
        if int(err.item()) != 0:
            raise RuntimeError("read_probe: a wait timed out")
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in times)
        med = statistics.median(us)
        rows.append({"bytes": nbytes, "us_median": round(med, 2), "us_min": round(us[0], 2),
                     "GBps_median": round(nbytes / (med * 1e-6) / 1e9, 1)})
        del buf
    print(json.dumps({"probe": "read_ceiling", "ctas_per_sm": args.probe_ctas_per_sm,
                      "chunk_bytes": args.probe_chunk, "stages": args.probe_stages, "steps": args.steps,
                      "l2": "flushed before each launch (write then read of 2x L2 size)", "rows": rows}),
          flush=True)


def main():
    args = parse()
    if args.clock_sampler is not None:
        raise SystemExit(nvml_sampler_main(args.clock_sampler, args.clock_interval_ms))
    if args.read_probe:
        return run_read_probe(args)
    world, rank, local = dist_env()
    from synth.workloads import materialize, workload
    if args.tq > 1:
        p = workload(args.workload, data=False)
        p.tq = args.tq
        p.name = f"{p.name}_tq{args.tq}"
        materialize(p)
    else:
        p = workload(args.workload)
    kv_bytes_gqa = p.kv_bytes
    if args.fa2_style:
        import numpy as np
        G = p.Hq // p.Hkv
        axis = 1 if p.layout == 0 else 1
        p.k = np.repeat(p.k, G, axis=axis)
        p.v = np.repeat(p.v, G, axis=axis)
        p.Hkv = p.Hq
        p.num_splits = 1
        p.name = f"{p.name}_fa2style"

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo" if args.impl == "reference" else "nccl")

    if args.impl == "reference":
        line = run_reference(args, p, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch

    import split_kv_decode_decoding_gb300 as da
    da.build()
    da.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    split_len = 0
    if args.varsplit:
        split_len, S = da.varsplit_plan(p.B, p.Hq * p.tq, p.Hkv, p.D, p.total_kv, max(p.lens))
        if args.split_len:
            split_len = args.split_len
            S = min(da.DA_MAX_SPLITS, -(-max(p.lens) // split_len))
    else:
        S = args.splits or p.num_splits or da.num_splits(p.B, p.Hq * p.tq, p.Hkv, p.D, min(p.lens),
                                                          max(p.lens))
    if args.fa2_style:
        S = 1
    hq, hk, hv, hcu = problem_tensors(p, dev)
    q, k, v, cu = hq.to(dev), hk.to(dev), hv.to(dev), hcu.to(dev)
    out = torch.empty(*p.q.shape, dtype=q.dtype, device=dev)
    ws = da.alloc_workspace(p.B * p.tq, p.Hq, p.D, S, device=dev, stream=stream)

    if args.cuda_core_math and (split_len or p.tq > 1 or p.Hq // p.Hkv > 8):
        raise SystemExit("--cuda-core-math takes uniform splits, one query token and G <= 8")
    if args.tmem_math and (split_len or args.cuda_core_math or (p.Hq // p.Hkv) * p.tq <= 8
                           or p.Hq // p.Hkv > 32):
        raise SystemExit("--tmem-math takes uniform splits and G * T_q > 8 with G <= 32")
    q_main, k_main, v_main, cu_main = q, k, v, cu
    out4 = out.view(p.B, p.tq, p.Hq, p.D)

    def call(bufs=None):
        # bufs: another (q, k, v, cu) set of device inputs (the end-to-end steps alternate two)
        q, k, v, cu = bufs if bufs is not None else (q_main, k_main, v_main, cu_main)
        if args.tmem_math:
            da.decode_attn_splitkv_multiquery_tmem(q.view(p.B, p.tq, p.Hq, p.D), k, v, cu, out4, ws,
                                                   num_splits=S, scale=p.scale, layout=p.layout,
                                                   stream=stream)
        elif args.cuda_core_math:
            da.decode_attn_splitkv_partial_cuda_core(q, k, v, cu, ws, num_splits=S, scale=p.scale,
                                                     layout=p.layout, stream=stream)
            if S > 1:
                da.decode_attn_splitkv_combine(out, ws, num_splits=S, stream=stream)
        elif split_len and p.tq > 1:
            da.decode_attn_splitkv_multiquery_varsplit(q, k, v, cu, out, ws, split_len=split_len, max_splits=S,
                                                       scale=p.scale, layout=p.layout, stream=stream)
        elif split_len:
            da.decode_attn_splitkv_varsplit(q, k, v, cu, out, ws, split_len=split_len, max_splits=S,
                                            scale=p.scale, layout=p.layout, stream=stream)
        elif p.tq > 1:
            da.decode_attn_splitkv_multiquery(q, k, v, cu, out, ws, num_splits=S, scale=p.scale,
                                              layout=p.layout, stream=stream)
        else:
            da.decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale,
                                   layout=p.layout, stream=stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # L2 flush: write one buffer twice the L2 size, then read another one, so the
    # timed kernel starts with none of its inputs cached and no dirty lines to write back
    flush_w = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)

    def flush():
        if not args.no_flush:
            flush_w.fill_(1)
            flush_r.sum()

    def step(ev0=None, ev1=None):
        # one public call: split kernel + combine kernel (chained by programmatic launch)
        flush()
        if ev0 is not None:
            ev0.record(stream)
        call()
        if ev1 is not None:
            ev1.record(stream)

    def split_step(ev0, ev1):
        # the split kernel alone, for its roofline; the combine follows untimed
        if split_len or p.tq > 1 or args.tmem_math:
            return step(ev0, ev1)   # these modes have no split-only entry point: time the call
        flush()
        ev0.record(stream)
        partial = (da.decode_attn_splitkv_partial_cuda_core if args.cuda_core_math
                   else da.decode_attn_splitkv_partial)
        partial(q, k, v, cu, ws, num_splits=S, scale=p.scale, layout=p.layout, stream=stream)
        ev1.record(stream)
        da.decode_attn_splitkv_combine(out, ws, num_splits=S, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        if da.decode_attn_splitkv_get_error(ws, stream=stream) != 0:
            raise RuntimeError("device error flag set during warm-up")
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        k_split = max(1, args.steps // 2)
        evk = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(k_split)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local) if not args.no_clocks else None
        if sampler:
            sampler.__enter__()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            step(*evs[i])
        for i in range(k_split):
            split_step(*evk[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        if sampler:
            sampler.__exit__(None, None, None)
        if world > 1:
            torch.distributed.barrier()
    # back-to-back calls, no flush between them (after the timed region, not part of it):
    # what a decode loop sees; the inputs stay in HBM only when they exceed the L2
    n_b2b = min(args.steps, 200)
    with torch.cuda.stream(stream):
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        flush()
        b0.record(stream)
        for _ in range(n_b2b):
            call()
        b1.record(stream)
        torch.cuda.synchronize(dev)
    b2b_ms = b0.elapsed_time(b1) / n_b2b
    if da.decode_attn_splitkv_get_error(ws, stream=stream) != 0:
        raise RuntimeError("device error flag set during the timed steps")
    step_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps)]
    split_ms = [evk[i][0].elapsed_time(evk[i][1]) for i in range(k_split)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    mean_step_ms = total_ms / args.steps
    value = world * kv_bytes_gqa / (mean_step_ms * 1e-3) / 1e9

    # ---- end to end through the public call, host buffers, copies inside each step
    e2e = None
    if args.e2e_steps > 0 and not (args.cuda_core_math or args.tmem_math):
        pq, pk, pv, pcu = hq.pin_memory(), hk.pin_memory(), hv.pin_memory(), hcu.pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        ncs = max(1, args.e2e_copy_streams)
        copy_streams = [torch.cuda.Stream(device=dev) for _ in range(ncs)]
        # Two sets of device inputs, used by alternate steps: a step's host-to-device
        # copies go into the set the previous step's call is not reading, so they run
        # while that call runs. Every step still copies all of its inputs in.
        nbuf = max(1, min(2, args.e2e_buffers))
        sets = [(q, k, v, cu)] + [tuple(torch.empty_like(t) for t in (q, k, v, cu)) for _ in range(nbuf - 1)]
        # K and V of each set cut into ncs pieces each, one piece of each per copy stream
        pieces = []
        for qx, kx, vx, cux in sets:
            ps = []
            for dst, src in ((kx, pk), (vx, pv)):
                fd, fs = dst.view(-1), src.view(-1)
                n = fd.numel()
                for i in range(ncs):
                    a_, b_ = n * i // ncs, n * (i + 1) // ncs
                    ps.append((i, fd[a_:b_], fs[a_:b_]))
            pieces.append(ps)
        read_done = [None] * nbuf   # per set: the event after the last call that read it
        step_no = [0]

        def e2e_step():
            si = step_no[0] % nbuf
            step_no[0] += 1
            qx, kx, vx, cux = sets[si]
            joins = []
            for i, cs in enumerate(copy_streams):
                if read_done[si] is not None:
                    cs.wait_event(read_done[si])   # the set's previous reader is done with it
                with torch.cuda.stream(cs):
                    for j, d_, s_ in pieces[si]:
                        if j == i:
                            d_.copy_(s_, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                joins.append(ev)
            qx.copy_(pq, non_blocking=True)
            cux.copy_(pcu, non_blocking=True)
            for ev in joins:
                stream.wait_event(ev)
            call((qx, kx, vx, cux))
            done = torch.cuda.Event()
            done.record(stream)
            read_done[si] = done
            hout.copy_(out, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for cs in copy_streams:
                cs.wait_event(e0)   # no copy of the timed steps starts before the clock
            for _ in range(args.e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in (pq, pk, pv, pcu))
        e2e = {"value": round(world * p.kv_bytes / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "api": "decode_attn_splitkv (C ABI), pinned host buffers",
               "copy_streams": ncs, "input_sets": nbuf}

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    per_call = 1 if (S == 1 and not split_len) else 2          # one split writes the output itself
    per_split_step = per_call if (split_len or p.tq > 1 or args.tmem_math) else 2
    split_mean_ms = sum(split_ms) / len(split_ms)
    ws_bytes = p.B * p.tq * p.Hq * S * (p.D + 1) * 4
    q_bytes = p.B * p.tq * p.Hq * p.D * 2
    alg_bytes = p.kv_bytes + q_bytes + 4 * (p.B + 1) + ws_bytes
    achieved = alg_bytes / (split_mean_ms * 1e-3) / 1e9
    traffic, traffic_src = (None, None) if (args.cuda_core_math or args.tmem_math) else \
        recorded_traffic(p.name, S)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_step_ms, 5),
        "us_per_call": round(mean_step_ms * 1e3, 2),
        "us_per_call_median": round(statistics.median(step_ms) * 1e3, 2),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": p.dtype, "data": "synthetic (seeded N(0,1), rounded to the input dtype)",
        "config": {**workload_config(p, S),
                   "products": ("CUDA-core fp32 FMA (comparison arm)" if args.cuda_core_math
                                else "tcgen05 with tensor memory (comparison arm)" if args.tmem_math
                                else "tensor-core mma.sync m16n8k16"),
                   **({"split_mode": "per-sequence", "split_len": split_len, "max_splits": S}
                      if split_len else {"split_mode": "uniform"})},
        "roofline": {"kernel": ("split_kernel_tc+combine_kernel" if args.tmem_math
                                else "split_kernel" if not (split_len or p.tq > 1)
                                else "split_kernel+combine_kernel"),
                     "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic, "traffic_source": traffic_src,
                     "alg_bytes_per_launch": alg_bytes,
                     "launch_us_mean": round(split_mean_ms * 1e3, 2),
                     "launches_timed": k_split,
                     **({"combine_us_mean_derived": round((mean_step_ms - split_mean_ms) * 1e3, 2)}
                        if per_call == 2 and not (split_len or p.tq > 1 or args.tmem_math) else {})},
        "back_to_back": {"us_per_call": round(b2b_ms * 1e3, 2),
                         "value": round(world * kv_bytes_gqa / (b2b_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                         "calls": n_b2b, "inputs_exceed_l2": p.kv_bytes > l2,
                         "note": "calls back to back without an L2 flush, after the timed region"},
        "e2e": e2e,
        "gpu_launches": per_call * args.steps + per_split_step * k_split,
        "model_us": (round(da.model_us(p.lens, p.Hq, p.Hkv, p.D, S,
                                       torch.cuda.get_device_properties(dev).multi_processor_count,
                                       T_q=p.tq), 1)
                     if not (split_len or args.fa2_style or args.cuda_core_math or args.tmem_math) else None),
        "wall_s_timed_region": round(t_wall, 3),
    }
    if sampler:
        line["clocks"] = sampler.summary()
    if not args.no_cpu_baseline and world == 1:
        gbs, cores, desc, _ = cpu_oracle_sample(p)
        gbs1, desc1 = cpu_oracle_one_thread(p)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle", "sample": desc,
                                "one_thread": {"value": round(gbs1, 4), "unit": "GB/s", "sample": desc1}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
