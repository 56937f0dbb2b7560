"""Calibrate the library's GB300 time model and the split-count picker on this GPU.

    python -m split_kv_decode_decoding_gb300.calibrate sweep --out sweep.json [--workloads a,b | --multiquery]
        call time against split count for the named workloads (GPU): L2 flushed before
        every call (a write of twice the L2 size, then a read of another such buffer),
        CUDA events on the launching stream, median of --reps calls; --multiquery sweeps
        the workloads with 2 or 4 new tokens per sequence
    python -m split_kv_decode_decoding_gb300.calibrate fit sweep.json [more.json ...]
        least-squares fit (in log time) of the 8 model parameters of
        decode_attn_splitkv_model_us to the calls within 30 % of their workload's
        fastest split count (CPU); prints the parameters and the errors
    python -m split_kv_decode_decoding_gb300.calibrate fa2 --out fa2.json
        FlashAttention-2-style decode (K/V repeated per query head, one split) against
        split-KV decode with the picker's split count, on the CodeLlama-34B shapes (GPU)

Inputs come from the seeded synthetic workloads (synth.workloads); run from the
repository root.
"""
from __future__ import annotations

import argparse
import json
import math
import statistics
import sys

from . import (alloc_workspace, build, decode_attn_splitkv, decode_attn_splitkv_get_error,
               decode_attn_splitkv_multiquery, decode_attn_splitkv_varsplit, load, model_us, num_splits)

SPLITS = [1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 19, 24, 32, 38, 48, 64, 76, 96, 128, 192, 256]
WORKLOADS = [
    "mha_bhsd", "qwen_varlen", "codellama_B256_S256", "codellama_B64_S1024", "codellama_B16_S4096",
    "codellama_B4_S16384", "codellama_B1_S65536", "codellama_B1_S131072", "llama_S1024_B1", "llama_S1024_B16",
    "llama_S8192_B1", "llama_S8192_B16", "llama_S32768_B1", "llama_S32768_B16", "llama_S131072_B1",
    "llama_S131072_B16", "llama_skewed"]
# several new tokens per sequence (decode_attn_splitkv_multiquery), 8- and 16-column items
MULTIQUERY_WORKLOADS = [
    "qwen_varlen_tq2", "qwen_varlen_tq4", "llama_S8192_B16_tq2", "llama_S8192_B16_tq4", "llama_S32768_B16_tq2",
    "llama_S32768_B16_tq4", "llama_S131072_B1_tq4", "codellama_B16_S4096_tq2", "llama_S8192_B1_tq4"]


class _Timer:
    """Median CUDA-event time of a call, with the L2 flushed before each call."""

    def __init__(self, reps: int):
        import torch
        self.torch = torch
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stream = torch.cuda.Stream(device=self.dev)
        l2 = torch.cuda.get_device_properties(self.dev).L2_cache_size
        self.flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=self.dev)
        self.flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=self.dev)
        self.reps = reps

    def __call__(self, fn) -> float:
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(self.reps + 3)]
        with torch.cuda.stream(self.stream):
            for a, b in evs:
                self.flush_w.fill_(1)
                self.flush_r.sum()
                a.record(self.stream)
                fn()
                b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs[3:])   # the first three warm up


def _device_problem(p, dev):
    import numpy as np
    import torch
    dt = torch.float16 if p.dtype == "f16" else torch.bfloat16

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt).to(dev)

    return up(p.q), up(p.k), up(p.v), torch.from_numpy(p.cu.astype(np.int32)).to(dev)


def _workload(name: str):
    """A named workload; a `_tqN` suffix asks for N query tokens per sequence."""
    from synth.workloads import materialize, workload
    if "_tq" not in name:
        return workload(name)
    base, tq = name.rsplit("_tq", 1)
    p = workload(base, data=False)
    p.tq = int(tq)
    p.name = name
    return materialize(p)


def sweep(names, reps: int, out_path: str) -> dict:
    import torch
    build()
    load()
    timer = _Timer(reps)
    dev, st = timer.dev, timer.stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    for name in names:
        p = _workload(name)
        q, k, v, cu = _device_problem(p, dev)
        p.k = p.v = None
        out = torch.empty(*p.q.shape, dtype=q.dtype, device=dev)
        splits = [S for S in SPLITS if S <= max(1, min(p.lens))]
        ws = alloc_workspace(p.B * p.tq, p.Hq, p.D, max(splits), device=dev, stream=st)
        row = {"lens": p.lens, "B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "D": p.D, "tq": p.tq, "sms": sms,
               "picker": num_splits(p.B, p.Hq * p.tq, p.Hkv, p.D, min(p.lens), max(p.lens), sms), "t": {}}
        entry = decode_attn_splitkv if p.tq == 1 else decode_attn_splitkv_multiquery
        for S in splits:
            row["t"][str(S)] = round(timer(lambda S=S: entry(
                q, k, v, cu, out, ws, num_splits=S, scale=p.scale, layout=p.layout, stream=st)), 2)
        if p.tq == 1 and 2 * min(p.lens) <= max(p.lens):
            row["var"] = {}
            for sl in (512, 1024, 2048, 4096, 8192):
                ms = min(1024, -(-max(p.lens) // sl))
                ws2 = alloc_workspace(p.B, p.Hq, p.D, ms, device=dev, stream=st)
                row["var"][str(sl)] = round(timer(lambda sl=sl, ms=ms, ws2=ws2: decode_attn_splitkv_varsplit(
                    q, k, v, cu, out, ws2, split_len=sl, max_splits=ms, scale=p.scale, layout=p.layout,
                    stream=st)), 2)
                del ws2
        if decode_attn_splitkv_get_error(ws, stream=st) != 0:
            raise RuntimeError(f"device error flag set on {name}")
        res[name] = row
        best = min(row["t"].items(), key=lambda kv: kv[1])
        print(f"{name:22s} picker S={row['picker']} {row['t'].get(str(row['picker']))} us, "
              f"best S={best[0]} {best[1]} us", flush=True)
        with open(out_path, "w") as f:
            json.dump(res, f)
        del q, k, v, cu, out, ws
        torch.cuda.empty_cache()
    return res


def _log_err(args):
    params, pts = args
    load()
    e = 0.0
    for r, S, t in pts:
        p = model_us(r["lens"], r["Hq"], r["Hkv"], r["D"], S, r["sms"], r.get("tq", 1), params)
        if p <= 0:
            return 1e9
        e += (math.log(p) - math.log(t)) ** 2
    return e


def fit(paths, within: float = 1.3, workers: int = 8) -> dict:
    import multiprocessing as mp

    import numpy as np
    from scipy.optimize import minimize
    load()
    d = {}
    for path in ([paths] if isinstance(paths, str) else paths):
        d.update(json.load(open(path)))
    pts, allpts = [], []
    for name, r in d.items():
        best = min(r["t"].values())
        for S, t in r["t"].items():
            allpts.append((name, r, int(S), t))
            if t <= within * best:
                pts.append((name, r, int(S), t))
    chunks = [[(r, S, t) for _, r, S, t in pts[i::workers]] for i in range(workers)]
    pool = mp.get_context("fork").Pool(workers)

    def loss(x):
        params = [math.exp(v) for v in x]
        return sum(pool.map(_log_err, [(params, c) for c in chunks]))

    x = [math.log(v) for v in (12.12, 1e-3, 76030, 7.727e6, 3.563, 6.607e5, 0.05334, 46900)]
    best = None
    for _ in range(3):
        res = minimize(loss, x if best is None else best.x, method="Nelder-Mead",
                       options={"maxiter": 3000, "xatol": 1e-4, "fatol": 1e-7})
        if best is None or res.fun < best.fun:
            best = res
    pool.close()
    params = [math.exp(v) for v in best.x]

    def err(sel):
        return np.array([abs(model_us(r["lens"], r["Hq"], r["Hkv"], r["D"], S, r["sms"], r.get("tq", 1), params) / t - 1)
                         for _, r, S, t in sel])
    e, ea = err(pts), err(allpts)
    out = {"params": params, "fitted_calls": len(pts), "measured_calls": len(allpts),
           "median_err": float(np.median(e)), "p90_err": float(np.percentile(e, 90)),
           "median_err_all": float(np.median(ea)), "p90_err_all": float(np.percentile(ea, 90))}
    print(json.dumps(out, indent=1))
    return out


def fa2(reps: int, out_path: str) -> dict:
    import torch
    from synth.workloads import CODELLAMA_SWEEP, workload
    build()
    load()
    timer = _Timer(reps)
    dev, st = timer.dev, timer.stream
    res = {}
    for b, s in CODELLAMA_SWEEP:
        p = workload(f"codellama_B{b}_S{s}")
        q, k, v, cu = _device_problem(p, dev)
        out = torch.empty(*p.q.shape, dtype=q.dtype, device=dev)
        S = num_splits(p.B, p.Hq, p.Hkv, p.D, min(p.lens), max(p.lens))
        ws = alloc_workspace(p.B, p.Hq, p.D, S, device=dev, stream=st)
        t_fd = timer(lambda: decode_attn_splitkv(q, k, v, cu, out, ws, num_splits=S, scale=p.scale,
                                                 layout=p.layout, stream=st))
        G = p.Hq // p.Hkv
        k_rep = k.repeat_interleave(G, dim=1).contiguous()
        v_rep = v.repeat_interleave(G, dim=1).contiguous()
        ws1 = alloc_workspace(p.B, p.Hq, p.D, 1, device=dev, stream=st)
        t_fa2 = timer(lambda: decode_attn_splitkv(q, k_rep, v_rep, cu, out, ws1, num_splits=1, scale=p.scale,
                                                  layout=p.layout, stream=st))
        res[f"{b}_{s}"] = {"B": b, "seqlen": s, "S": S, "fd_us": round(t_fd, 2), "fa2_us": round(t_fa2, 2)}
        print(json.dumps(res[f"{b}_{s}"]), flush=True)
        del q, k, v, cu, out, ws, k_rep, v_rep, ws1
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump(res, f, indent=1)
    return res


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="cmd", required=True)
    a = sub.add_parser("sweep")
    a.add_argument("--out", required=True)
    a.add_argument("--workloads", default=",".join(WORKLOADS))
    a.add_argument("--multiquery", action="store_true")
    a.add_argument("--reps", type=int, default=25)
    b = sub.add_parser("fit")
    b.add_argument("sweep_json", nargs="+")
    b.add_argument("--within", type=float, default=1.3)
    c = sub.add_parser("fa2")
    c.add_argument("--out", required=True)
    c.add_argument("--reps", type=int, default=40)
    args = ap.parse_args(argv)
    if args.cmd == "sweep":
        sweep(MULTIQUERY_WORKLOADS if args.multiquery else args.workloads.split(","), args.reps, args.out)
    elif args.cmd == "fit":
        fit(args.sweep_json, args.within)
    else:
        fa2(args.reps, args.out)


if __name__ == "__main__":
    sys.exit(main())
