"""Compile the CUDA library for sm_103a, in tree (no cmake): four translation units
compiled in parallel, then linked into one shared library."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, n) for n in
           ("decode_attn_splitkv.cu", "comparison_arms.cu", "picker.cpp", "time_model.cpp")]
HEADER = os.path.join(ROOT, "include", "decode_attn_splitkv.h")
LIB = os.path.join(PKG, "_build", "libdecode_attn_splitkv.so")
# the read-ceiling probe the benchmark times beside the decode call (not part of the library)
PROBE_SRC = os.path.join(CSRC, "read_probe.cu")
PROBE_LIB = os.path.join(PKG, "_build", "libread_probe.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return cand


def inputs() -> list:
    """Every file the library is built from (sources and headers)."""
    return SOURCES + [HEADER] + sorted(glob.glob(os.path.join(CSRC, "*.h")) +
                                       glob.glob(os.path.join(CSRC, "*.cuh")))


def build_probe(force: bool = False) -> str:
    """Compile the read-ceiling probe into its own small library."""
    os.makedirs(os.path.dirname(PROBE_LIB), exist_ok=True)
    if not force and os.path.exists(PROBE_LIB) and os.path.getmtime(PROBE_LIB) >= os.path.getmtime(PROBE_SRC):
        return PROBE_LIB
    tmp = PROBE_LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *NVCC_FLAGS, "-shared", "-o", tmp, PROBE_SRC], check=True)
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    newest = max(os.path.getmtime(f) for f in inputs())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(os.path.dirname(LIB), os.path.basename(s) + tag + ".o") for s in SOURCES]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose and src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)

    try:
        with ThreadPoolExecutor(len(SOURCES)) as ex:
            list(ex.map(compile_one, zip(SOURCES, objs)))
        tmp = LIB + tag
        subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                        "-Xcompiler", "-fPIC", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB
