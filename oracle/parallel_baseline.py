"""Loader for parallel_baseline.c -- BENCHMARK INFRASTRUCTURE ONLY (bench.py's CPU comparison line).

Not the oracle: see parallel_baseline.c.  Builds it with gcc -fopenmp into oracle/_build and
times it on a problem from workloads.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "parallel_baseline.c")
LIB = os.path.join(_HERE, "_build", "libparallel_baseline.so")


def build(out: str = LIB) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", out, SOURCE],
                   check=True)
    return out


def load() -> ctypes.CDLL:
    import oracle

    if not (os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SOURCE)
            and oracle._built_for_this_host(LIB)):
        build()
    lib = ctypes.CDLL(LIB)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.mrr_cpu_parallel_run.restype = ctypes.c_int
    lib.mrr_cpu_parallel_run.argtypes = [P, I64, I64, P, ctypes.c_int, I64, I64, P, I64, P,
                                         P, P, P, P, P, I64, ctypes.c_int]
    return lib


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run(lib, p, outs, threads: int) -> None:
    """One pass of the moves over problem p into the preallocated outs."""
    ptr = lambda a: None if a is None else a.ctypes.data
    st = lib.mrr_cpu_parallel_run(ptr(p.tokens), p.A, p.row_bytes, ptr(p.counts),
                                  int(p.counts.dtype == np.int64), p.N, p.E, ptr(p.scales),
                                  p.scale_row_bytes, ptr(p.topk), ptr(outs["tokens"]),
                                  ptr(outs["scales"]), ptr(outs["idx"]), ptr(outs["etn"]),
                                  ptr(outs["topk"]), p.idx_type, threads)
    if st != 0:
        raise RuntimeError("parallel CPU baseline failed to allocate")


def time_problem(p, budget_s: float):
    """GB/s (the op's algorithmic bytes) over repeated passes for about budget_s seconds."""
    lib = load()
    threads = host_threads()
    outs = {"tokens": np.empty(p.A * p.row_bytes, np.uint8),
            "scales": None if p.scales is None else np.empty(p.A * p.scale_row_bytes, np.uint8),
            "idx": np.empty(p.A, np.int32), "etn": np.empty(p.E, p.counts.dtype),
            "topk": None if p.topk is None else np.empty(p.A, np.float32)}
    run(lib, p, outs, threads)  # first touch of the outputs
    reps, t0 = 0, time.perf_counter()
    while True:
        run(lib, p, outs, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return p.algorithmic_bytes() * reps / el / 1e9, reps, el, threads, outs
