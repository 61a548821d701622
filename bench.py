#!/usr/bin/env python
"""Benchmark of the MoeReRoutingV2 re-routing step on GB300.

One step = one mrr_v2_run call over one batch: the whole hot path (count validation, both
offset scans, expert_token_num, the token / scale / top-k moves and the index) for the
workload A=16384, H=7168 int8 tokens, N=16 ranks x E=16 experts with the skewed count matrix
of the torch_npu.npu_moe_re_routing usage example (one cell holds 16129 of the 16384 rows),
fp32 per-token scales [A], no top-k weights, idx_type 0.

Prints ONE JSON line.  ``value`` is effective HBM GB/s: the algorithmic bytes (every input
byte read once, every output byte written once) per step over the device time per step, with
inputs resident in HBM.  Consecutive steps rotate over buffer sets whose combined footprint is
several times the L2 size, so no step reads what an earlier step left in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--impl gb300|reference]

--impl reference times the CPU oracle (a plain loop restatement of the op, single-threaded)
on the same workload: each step is a bounded row sample of it, so the run ends in minutes.
Multi-GPU (torchrun, one rank per GPU) runs independent replicas: the op has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (read+write) and % of GB300 peak; tokens/sec at A=16384,H=7168"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, help="workload 1..5 (2 is the headline)")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--op", choices=["route", "unroute", "multi", "push", "gating"], default="route",
                    help="route: rank-major -> expert-major (the op); unroute: the inverse move; "
                         "multi: the op reading each source rank's rows from a buffer of its own; "
                         "push: one sender writing the workload's rows into N receivers' buffers "
                         "(mrr_v2_push; the receivers are this GPU's memory); "
                         "gating: the upstream gating top-k op (--config 1, 2 or 3)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU oracle baseline budget (seconds of oracle work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-detail", action="store_true",
                    help="skip the batch spread, unrotated and CUDA-graph timings")
    ap.add_argument("--multi-layout", choices=["separate", "slots"], default="separate",
                    help="--op multi: one allocation per source rank, or one receive buffer with a "
                         "slot of the largest rank's rows per rank")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time only the chosen workload (by default workload 2 is followed by 3, 4 and 5)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The maximum of ``value`` over all ranks (the slowest rank sets the job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_gbs(world: int, bytes_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job GB/s: every rank moved ``bytes_per_step`` per step; time is the max over ranks."""
    return world * bytes_per_step * steps / (elapsed_ms * 1e-3) / 1e9


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo", encoding="utf-8"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_text(rel: str) -> bytes:
    """A source file's code: its text without // comments, trailing blanks and empty lines, so
    that a change to comments alone leaves the hash (and a profile's claim to it) unchanged.  The
    hashed sources hold no "//" inside a string literal."""
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        lines = (re.sub(r"//.*", "", line).rstrip() for line in f)
        return "\n".join(line for line in lines if line).encode()


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("moe_expert_token_gb300/csrc/mrr_v2.cu", "moe_expert_token_gb300/csrc/ptx.cuh",
                "moe_expert_token_gb300/csrc/ws_layout.h"):
        h.update(code_text(rel))
    return h.hexdigest()[:16]


def push_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("moe_expert_token_gb300/csrc/mrr_push.cu", "moe_expert_token_gb300/csrc/mrr_shape.h",
                "moe_expert_token_gb300/csrc/ptx.cuh", "moe_expert_token_gb300/csrc/ws_layout.h"):
        h.update(code_text(rel))
    return h.hexdigest()[:16]


def profiled_traffic(config: int, op: str = "route"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    name = {"route": f"reroute_kernel_C{config}.md", "unroute": f"reroute_kernel_inverse_C{config}.md",
            "multi": f"reroute_kernel_multi_C{config}.md", "push": f"push_kernel_C{config}.md"}.get(op)
    if name is None:   # no committed summary for this op
        return None
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not src or not tr or src.group(1) != (push_source_hash() if op == "push" else kernel_source_hash()):
        return None
    return int(tr.group(1))


GATING_PROFILES = {1: "gating_kernel_T16384_e384_top6.md", 2: "gating_kernel_T16384_e256_grouped_top8.md",
                   3: "gating_kernel_T16384_e384_fp32_top6.md"}


def gating_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("moe_expert_token_gb300/csrc/gating.cu", "moe_expert_token_gb300/csrc/gating_kernel.cuh",
                "moe_expert_token_gb300/csrc/gating_f16.cu", "moe_expert_token_gb300/csrc/gating_bf16.cu",
                "moe_expert_token_gb300/csrc/gating_f32.cu", "moe_expert_token_gb300/csrc/ptx.cuh"):
        h.update(code_text(rel))
    return h.hexdigest()[:16]


def profiled_gating_field(config: int, field: str):
    """An integer field (e.g. DRAM bytes per launch) of the gating kernel's committed ncu summary
    for workload `config`, if that summary was taken on the current kernel source."""
    try:
        text = open(os.path.join(ROOT, "profiles", GATING_PROFILES[config]), encoding="utf-8").read()
    except (OSError, KeyError):
        return None
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    val = re.search(field + r":\s*([0-9]+)", text)
    if not src or not val or src.group(1) != gating_source_hash():
        return None
    return int(val.group(1))


def profiled_gating_traffic(config: int):
    """DRAM bytes per launch of the gating kernel from its committed ncu summary, if current."""
    return profiled_gating_field(config, "traffic_bytes_per_launch")


SM_COUNT = 152          # GB300: 2 dies x 76 SMs
ISSUE_PER_SM = 4        # one warp instruction per cycle from each of an SM's 4 schedulers


def gating_issue_roofline(config: int, mean_launch_us: float, clocks: dict):
    """The gating kernel is bound by instruction issue, not HBM: its warp instructions per launch
    (from the committed ncu summary, if current) over the launch time, against the GPU's issue
    peak (SMs x 4 schedulers x the SM clock sampled during the run, else the 2070 MHz maximum)."""
    inst = profiled_gating_field(config, "warp_instructions_per_launch")
    if inst is None or mean_launch_us <= 0:
        return None
    mhz = clocks.get("sm_mhz") or 2070.0
    peak = SM_COUNT * ISSUE_PER_SM * mhz * 1e6
    achieved = inst / (mean_launch_us * 1e-6)
    return {"bound": "issue", "achieved": achieved, "peak": peak, "unit": "warp instructions/s",
            "frac": achieved / peak, "warp_instructions_per_launch": inst, "sm_mhz": mhz,
            "source": "profiles/" + GATING_PROFILES[config]}


class ClockSampler:
    """nvidia-smi clock / throttle samples, taken while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.rows = []
        self.proc = None
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        lo, hi = self.t_start - 0.05, self.t_end + 0.05
        win = [r for t, r in self.rows if lo <= t <= hi]
        window = "timed"
        if len(win) < 3:          # a short timed region: fall back to the whole run
            win = [r for _, r in self.rows]
            window = "run (timed region shorter than the sampling period)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in win:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for k, n in enumerate(names):
                if len(r) > 5 + k and r[5 + k].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(win), "window": window}


# ----------------------------------------------------------------------------- sampling for the CPU legs

def row_sample(p, frac: float):
    """A smaller problem of the same kind: the first A' rows, counts scaled to sum to A'."""
    import numpy as np

    if frac >= 1.0:
        return p
    N, E = p.counts.shape
    A2 = max(N * E, int(p.A * frac))
    c = p.counts.astype(np.int64)
    extra = (c - 1) * (A2 - N * E) // max(1, p.A - N * E)
    c2 = 1 + extra
    c2.flat[int(np.argmax(c2))] += A2 - int(c2.sum())
    import copy

    q = copy.copy(p)
    q.A = A2
    q.counts = c2.astype(p.counts.dtype)
    q.tokens = p.tokens[:A2]
    q.scales = None if p.scales is None else p.scales[:A2]
    q.topk = None if p.topk is None else p.topk[:A2]
    return q


def op_bytes(p, op: str) -> int:
    """Algorithmic bytes of one step.  The inverse move writes no index and no per-expert counts;
    the multi-source form moves the same bytes as the op (plus N pointers per table, not counted);
    the push form writes the index but no per-expert counts, and reads two int64 offset tables."""
    if op in ("route", "multi"):
        return p.algorithmic_bytes()
    if op == "push":
        return p.algorithmic_bytes() - p.E * p.counts.dtype.itemsize + 2 * 8 * p.N * p.E
    return p.algorithmic_bytes() - 4 * p.A - p.E * p.counts.dtype.itemsize


def oracle_step(p, op: str, lib):
    import oracle

    if op in ("route", "multi", "push"):   # multi: the oracle of the concatenation (the same rows);
        return oracle.run_problem(p, lib=lib)  # push: the same rows placed expert-major
    # the workload's payloads stand for the expert-major rows the inverse move reads
    return oracle.unroute(p.tokens, p.counts, permute_scales=p.scales, permute_topk=p.topk, lib=lib)


def time_oracle(p, budget_s: float, op: str = "route", max_reps: int = 1000):
    """Run the oracle on ``p`` repeatedly for about ``budget_s`` seconds; (GB/s, reps, s)."""
    import oracle

    lib = oracle.load()
    oracle_step(p, op, lib)  # warm (page in the library and the inputs)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(p, op, lib)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    return op_bytes(p, op) * reps / el / 1e9, reps, el


def config_dict(p, k, extra=None, op="route"):
    name = {"route": p.name, "unroute": "inverse move of " + p.name,
            "multi": p.name + ", each source rank's rows in a buffer of their own",
            "push": p.name + ", pushed by one sender into the N receivers' expert-major buffers "
                             "(this GPU's memory)"}[op]
    d = {"workload": name, "op": op,
         "A": p.A, "H": p.H, "N": p.N, "E": p.E, "token_dtype": p.token_dtype,
         "count_dtype": str(p.counts.dtype), "scales": p.scale_layout, "scale_cols": p.scale_cols,
         "topk": p.topk is not None, "idx_type": p.idx_type, "expert_token_num_type": 1,
         "bytes_per_step": op_bytes(p, op)}
    d.update(extra or {})
    return d


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import workloads

    p = workloads.config(args.config)
    # size each step so that warmup + steps take about two minutes of oracle work at most
    t_full = time.perf_counter()
    import oracle

    lib = oracle.load()
    oracle_step(p, args.op, lib)
    t_full = time.perf_counter() - t_full
    frac = min(1.0, 120.0 / max(1e-9, t_full * (args.steps + args.warmup)))
    q = row_sample(p, frac)
    for _ in range(args.warmup):
        oracle_step(q, args.op, lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(q, args.op, lib)
    el = time.perf_counter() - t0
    value = op_bytes(q, args.op) * args.steps / el / 1e9
    sample = f"first {q.A} of {p.A} rows per step (counts scaled to sum to {q.A})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic", "config": config_dict(p, args.config, {"sample_rows": q.A}, args.op),
        "tokens_per_s": q.A * args.steps / el,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

class RouteSetup:
    """One workload on one GPU: its plan, rotating device buffer sets, and the C-ABI call of one
    step (mrr_v2_run, or mrr_v2_unroute for the inverse move) with its arguments resolved."""

    def __init__(self, p, op, dev, local_rank, multi_layout="separate"):
        import numpy as np
        import torch
        import moe_expert_token_gb300.mrr_v2 as m

        self.p, self.op, self.dev, self.m = p, op, dev, m
        code = m.DTYPE_CODES[p.token_dtype]
        sl = m.SCALE_CODES[p.scale_layout]
        A, H, N, E = p.A, p.H, p.N, p.E
        i64 = int(p.counts.dtype == np.int64)
        if op == "push":   # no plan: one launch of the push kernel (plain copies, 3 CTAs per SM)
            import types

            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            st, plan = m.MRR_OK, types.SimpleNamespace(path=2, grid=min(3 * sms, -(-A // 8)), block=256,
                                                       chunk_bytes=0, stages=0, fuse_scan=1, workspace_bytes=4096)
        elif op in ("route", "multi"):
            st, plan = m.mrr_v2_plan(A, H, code, N, E, i64, sl, p.scale_cols, p.topk is not None, 1,
                                     p.idx_type, local_rank)
        else:
            st, plan = m.mrr_v2_unroute_plan(A, H, code, N, E, i64, sl, p.scale_cols, p.topk is not None,
                                             local_rank)
        if st != m.MRR_OK:
            raise SystemExit(m.mrr_status_str(st))
        self.plan = plan
        self.launches_per_step = 1 if plan.fuse_scan else 2
        self.bytes_step = op_bytes(p, op)

        def dev_bytes(arr):
            if arr is None:
                return None
            return torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1).copy()).to(dev)

        # buffer sets: enough that consecutive steps never hit in L2
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.R = R = max(2, -(-4 * self.l2 // self.bytes_step))
        host_in = {"tokens": p.tokens, "counts": p.counts, "scales": p.scales, "topk": p.topk}
        inv = op == "unroute"   # the inverse move writes no index and no per-expert counts
        bounds = np.concatenate([[0], np.cumsum(p.counts.astype(np.int64).sum(axis=1))])
        self.sets = []
        for _ in range(R):
            s = {k: dev_bytes(v) for k, v in host_in.items()}
            if op == "multi":
                # one device buffer per source rank for each payload, and the tables of their
                # addresses; the single buffers above are dropped
                rows = np.diff(bounds)
                cap = int(rows.max())
                for key, rb in (("tokens", p.row_bytes), ("scales", p.scale_row_bytes), ("topk", 4)):
                    if s[key] is None:
                        s["tab_" + key] = None
                        continue
                    if multi_layout == "slots":   # one receive buffer, rank i's slot at i * cap rows
                        slab = torch.empty(N * cap * rb, dtype=torch.uint8, device=dev)
                        parts = [slab[i * cap * rb:i * cap * rb + int(rows[i]) * rb] for i in range(N)]
                        for i, t in enumerate(parts):
                            t.copy_(s[key][bounds[i] * rb:bounds[i + 1] * rb])
                        s["slab_" + key] = slab
                    else:
                        parts = [s[key][bounds[i] * rb:bounds[i + 1] * rb].clone() for i in range(N)]
                    for i, t in enumerate(parts):
                        s[f"{key}@{i}"] = t
                    s["tab_" + key] = torch.tensor([t.data_ptr() for t in parts], dtype=torch.int64, device=dev)
                    s[key] = None
                s["rows"] = torch.tensor(np.full(N, cap) if multi_layout == "slots" else rows, dtype=torch.int64,
                                         device=dev)
            if op == "push":
                # N receivers, each holding this sender's rows for it expert-major: segment (r, j)
                # at DstOffset = the rows of r's experts before j (also the segment's rank-major row)
                c64 = p.counts.astype(np.int64)
                rows_r = c64.sum(axis=1)
                offs = np.concatenate([np.zeros((N, 1), np.int64), np.cumsum(c64, axis=1)[:, :-1]], axis=1)
                s["dst_off"] = torch.from_numpy(np.ascontiguousarray(offs)).to(dev)
                s["out_rows"] = torch.from_numpy(rows_r.copy()).to(dev)
                for key, rb in (("tok", p.row_bytes), ("sc", p.scale_row_bytes), ("tk", 4), ("idx", 4)):
                    if (key == "sc" and p.scales is None) or (key == "tk" and p.topk is None):
                        s["tab_" + key] = None
                        continue
                    parts = [torch.empty(int(rows_r[r]) * rb, dtype=torch.uint8, device=dev) for r in range(N)]
                    for r, t in enumerate(parts):
                        s[f"{key}@{r}"] = t
                    s["tab_" + key] = torch.tensor([t.data_ptr() for t in parts], dtype=torch.int64, device=dev)
                s["ws"] = torch.empty(4096, dtype=torch.uint8, device=dev)
                self.sets.append(s)
                continue
            s["out_tokens"] = torch.empty(A * p.row_bytes, dtype=torch.uint8, device=dev)
            s["out_scales"] = (None if p.scales is None
                               else torch.empty(A * p.scale_row_bytes, dtype=torch.uint8, device=dev))
            s["out_topk"] = None if p.topk is None else torch.empty(4 * A, dtype=torch.uint8, device=dev)
            s["idx"] = None if inv else torch.empty(A, dtype=torch.int32, device=dev)
            s["etn"] = None if inv else torch.empty(E * p.counts.dtype.itemsize, dtype=torch.uint8, device=dev)
            s["ws"] = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
            self.sets.append(s)
        lib = m.load_library()
        P = lambda t: None if t is None else t.data_ptr()
        if op == "route":
            self.fn = lib.mrr_v2_run
            self.args = [(P(s["tokens"]), code, A, H, P(s["counts"]), i64, N, E, P(s["scales"]), sl,
                          p.scale_cols, P(s["topk"]), P(s["out_tokens"]), P(s["out_scales"]), P(s["idx"]),
                          P(s["etn"]), P(s["out_topk"]), 1, p.idx_type, P(s["ws"]), s["ws"].numel())
                         for s in self.sets]
        elif op == "push":
            self.fn = lib.mrr_v2_push
            self.args = [(P(s["tokens"]), P(s["scales"]), P(s["topk"]), code, A, H, P(s["counts"]), i64, N, E, sl,
                          p.scale_cols, P(s["dst_off"]), P(s["dst_off"]), P(s["tab_tok"]), P(s["tab_sc"]),
                          P(s["tab_tk"]), P(s["tab_idx"]), P(s["out_rows"]), P(s["ws"]), s["ws"].numel())
                         for s in self.sets]
        elif op == "multi":
            self.fn = lib.mrr_v2_run_multi
            self.args = [(P(s["tab_tokens"]), P(s["tab_scales"]), P(s["tab_topk"]), P(s["rows"]), code, A, H,
                          P(s["counts"]), i64, N, E, sl, p.scale_cols, P(s["out_tokens"]), P(s["out_scales"]),
                          P(s["idx"]), P(s["etn"]), P(s["out_topk"]), 1, p.idx_type, P(s["ws"]), s["ws"].numel())
                         for s in self.sets]
        else:  # the inverse move: the "tokens" buffers hold the expert-major rows
            self.fn = lib.mrr_v2_unroute
            self.args = [(P(s["tokens"]), code, A, H, P(s["counts"]), i64, N, E, P(s["scales"]), sl,
                          p.scale_cols, P(s["topk"]), P(s["out_tokens"]), P(s["out_scales"]), P(s["out_topk"]),
                          P(s["ws"]), s["ws"].numel())
                         for s in self.sets]
        self.set_index = {id(s): i for i, s in enumerate(self.sets)}

    def launch(self, s, on_stream):
        """One step on ``on_stream``: the C-ABI call on buffer set ``s``."""
        st = self.fn(*self.args[self.set_index[id(s)]], on_stream.cuda_stream)
        if st != self.m.MRR_OK:
            raise RuntimeError(self.m.mrr_status_str(st))

    def gate(self, stream):
        """Untimed correctness gate on every buffer set: device status and a permutation check."""
        import torch

        m = self.m
        for s in self.sets:
            self.launch(s, stream)
            st = m.mrr_v2_read_status(s["ws"].data_ptr(), s["ws"].numel(), stream.cuda_stream)
            if st != m.MRR_OK:
                raise RuntimeError(m.mrr_status_str(st))
        if self.op in ("route", "multi"):
            idx_sorted = torch.sort(self.sets[0]["idx"].to(torch.int64)).values
            assert torch.equal(idx_sorted, torch.arange(self.p.A, device=self.dev)), "index is not a permutation"

    def check_status(self, stream):
        m = self.m
        for s in self.sets:
            st = m.mrr_v2_read_status(s["ws"].data_ptr(), s["ws"].numel(), stream.cuda_stream)
            if st != m.MRR_OK:
                raise RuntimeError(m.mrr_status_str(st))


HOLD_CYCLES = 600_000   # about 0.3 ms at the 2070 MHz maximum SM clock


def hold_stream(stream):
    """Queue a bounded device-side sleep (HOLD_CYCLES SM cycles) on `stream`.  Placed after the
    synchronize that opens a timed region and before its start event, it keeps the stream busy
    while the host makes its first calls after the synchronize, so that the region begins with
    the first launch already queued rather than waiting on the host (the blocking-kernel method
    of GPU benchmark harnesses).  The sleep itself lies before the start event."""
    import torch

    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)


def timed_steps(setup, K, W, stream, dev, dist=None, clocks=None):
    """W warm-up steps, then exactly K steps between two CUDA events on the launching stream,
    bracketed by a barrier and a device synchronize on both sides.  The warm-up runs directly
    before the timed region (nothing idles the GPU or the host in between), and hold_stream
    queues a short device sleep ahead of the start event.  An extra event after the first timed
    step shows how long that step took from the start of the region.
    Returns (region ms, first step us)."""
    import torch

    sets, R, fn, args = setup.sets, setup.R, setup.fn, setup.args
    h = stream.cuda_stream
    for k in range(W):
        setup.launch(sets[k % R], stream)
    t_begin, t_first, t_end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.t_start = time.time()
    hold_stream(stream)
    # only our launches run on this stream between the two events, back to back
    t_begin.record(stream)
    for k in range(K):
        st = fn(*args[k % R], h)
        if k == 0:
            t_first.record(stream)
        if st != 0:
            raise RuntimeError(setup.m.mrr_status_str(st))
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.t_end = time.time()
    if dist is not None:
        dist.barrier()
    return t_begin.elapsed_time(t_end), t_begin.elapsed_time(t_first) * 1e3


OTHER_CONFIGS = (3, 4, 5)
STEADY_K = 500


def run_gpu(args):
    import torch
    import workloads
    from moe_expert_token_gb300 import build as mbuild
    import moe_expert_token_gb300.mrr_v2 as m

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        mbuild.build()
    if dist is not None:
        dist.barrier()
    m.load_library()

    p = workloads.config(args.config)
    A = p.A
    setup = RouteSetup(p, args.op, dev, local_rank, args.multi_layout)
    plan, sets, R = setup.plan, setup.sets, setup.R
    bytes_step, launches_per_step = setup.bytes_step, setup.launches_per_step
    stream = torch.cuda.current_stream(dev)
    setup.gate(stream)

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)          # the sampler's first samples; the warm-up follows right before timing
    K = args.steps
    local_ms, first_us = timed_steps(setup, K, args.warmup, stream, dev, dist, clocks)
    time.sleep(0.2)
    clocks.stop()
    elapsed_ms = max_over_ranks(local_ms, dist, dev)
    value = throughput_gbs(world, bytes_step, K, elapsed_ms)
    ms_per_step = elapsed_ms / K
    # the timed region holds exactly K * launches_per_step of our launches back to back on one
    # stream: the average step (one launch for N*E <= 4096) is its length over K
    mean_launch_ms = local_ms / K
    achieved = bytes_step / (mean_launch_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    detail = None
    if not args.no_detail:
        detail = timing_detail(setup.launch, sets, stream, launches_per_step)
        detail["first_step_us"] = first_us
        detail["first_step_excess_us"] = first_us - detail["batch_us"]["p50"]
        setup.check_status(stream)   # the graph and unrotated runs left every set valid

    # end to end through the C ABI from pinned host buffers: H2D inputs, run, D2H outputs
    e2e = None
    if not args.no_e2e and args.op != "push":   # the push form's receivers are device buffers only
        e2e = run_e2e(args, p, sets, setup.launch, dev, bytes_step, world, dist)

    cpu = cpu_par = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, reps, el = time_oracle(p, args.cpu_seconds, args.op)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "cpu": cpu_model(), "kind": "oracle",
               "sample": f"the full workload, {reps} runs in {el:.1f} s, single thread"}
        if args.op == "route":
            cpu_par = time_cpu_parallel(p, min(args.cpu_seconds, 10.0))

    # the other large workloads, timed the same way in the same run (parity-tested elsewhere)
    others = None
    if args.op == "route" and args.config == 2 and not args.no_other_configs:
        del setup, sets
        torch.cuda.empty_cache()
        others = {}
        for k in OTHER_CONFIGS:
            q = workloads.config(k)
            su = RouteSetup(q, "route", dev, local_rank)
            su.gate(stream)
            ms_k, first_k = timed_steps(su, K, args.warmup, stream, dev, dist)
            ms_k = max_over_ranks(ms_k, dist, dev)
            gbs_k = throughput_gbs(world, su.bytes_step, K, ms_k)
            # the same launches over a longer region, where the first launch's start-up after
            # the synchronize weighs 1/STEADY_K instead of 1/K
            ms_s, _ = timed_steps(su, STEADY_K, args.warmup, stream, dev, dist)
            ms_s = max_over_ranks(ms_s, dist, dev)
            gbs_s = throughput_gbs(world, su.bytes_step, STEADY_K, ms_s)
            others[f"C{k}"] = {
                "workload": q.name, "value": gbs_k, "unit": "GB/s", "ms_per_step": ms_k / K,
                "pct_of_peak": 100.0 * gbs_k / world / peak, "frac": gbs_k / world / peak,
                "tokens_per_s": world * q.A * K / (ms_k * 1e-3), "bytes_per_step": su.bytes_step,
                "gpu_launches": K * su.launches_per_step, "first_step_us": first_k,
                "steady_state": {"steps": STEADY_K, "ms_per_step": ms_s / STEADY_K,
                                 "frac": gbs_s / world / peak},
                "path": {1: "bulk", 2: "vector"}[su.plan.path], "grid": su.plan.grid,
                "fused_scan": bool(su.plan.fuse_scan),
                "traffic": profiled_traffic(k, "route"),
                "l2": f"{su.R} rotating buffer sets, {su.R * su.bytes_step / 1e6:.0f} MB > 4x L2"}
            del su
            torch.cuda.empty_cache()

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded numpy draws shaped like the pages' workload)",
        "config": config_dict(p, args.config, op=args.op, extra={
            "l2": f"{R} rotating buffer sets, {R * bytes_step / 1e6:.0f} MB > 4x L2 ({setup_l2(dev) / 1e6:.0f} MB)",
            "path": {1: "bulk", 2: "vector"}[plan.path], "grid": plan.grid, "block": plan.block,
            "chunk_bytes": plan.chunk_bytes, "stages": plan.stages, "fused_scan": bool(plan.fuse_scan),
            "parallelism": f"replicas x{world}",
            **({"multi_layout": args.multi_layout} if args.op == "multi" else {})}),
        "pct_of_peak": 100.0 * value / world / peak,
        "tokens_per_s": world * A * K / (elapsed_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": profiled_traffic(args.config, args.op),
                     "kernel": "mrr_push::push_kernel" if args.op == "push" else "mrr::reroute_kernel",
                     "bytes_per_launch": bytes_step,
                     "mean_launch_us": mean_launch_ms * 1e3,
                     "timing": "CUDA events around the K back-to-back launches on the launching stream, a bounded "
                               "device sleep queued ahead of the start event so that the first launch is "
                               "already queued; per launch = region / K"},
        "cpu_baseline": cpu,
        "cpu_parallel": cpu_par,
        "timing_detail": detail,
        "e2e": e2e,
        "other_configs": others,
        "gpu_launches": K * launches_per_step,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def setup_l2(dev) -> int:
    import torch

    return torch.cuda.get_device_properties(dev).L2_cache_size


def time_cpu_parallel(p, budget_s: float):
    """The multi-core CPU comparison program (OpenMP blocks of per-segment memcpy, not the oracle)
    on the full workload, all host threads."""
    try:
        from oracle import parallel_baseline as pb

        gbs, reps, el, threads, _ = pb.time_problem(p, budget_s)
    except Exception as e:  # a host without OpenMP: report, do not fail the bench line
        return {"value": None, "error": str(e)[:200]}
    return {"value": gbs, "unit": "GB/s", "cores": threads, "cpu": cpu_model(),
            "kind": "openmp blocks of per-segment memcpy (a plain parallel program, not the oracle)",
            "sample": f"the full workload, {reps} runs in {el:.1f} s"}


def timing_detail(launch, sets, stream, launches_per_step, batches=20, per_batch=50):
    """Outside the timed region: the spread over batches of back-to-back launches (rotating sets),
    the same launches on one unrotated buffer set, and the launches captured once in a CUDA graph
    and replayed.  Microseconds per step."""
    import numpy as np
    import torch

    R = len(sets)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, n):
        torch.cuda.synchronize()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n

    per = []
    for j in range(batches):
        per.append(timed(lambda: [launch(sets[(j * per_batch + i) % R], stream) for i in range(per_batch)],
                         per_batch))
    unflushed = timed(lambda: [launch(sets[0], stream) for _ in range(per_batch)], per_batch)
    out = {"batches": batches, "launches_per_batch": per_batch,
           "batch_us": {q: float(np.percentile(per, v)) for q, v in (("p10", 10), ("p50", 50), ("p90", 90))},
           "unflushed_us": unflushed}
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=cap):
            for i in range(per_batch):
                launch(sets[i % R], cap)
        g.replay()
        reps = 10
        out["graph_us"] = timed(lambda: [g.replay() for _ in range(reps)], reps * per_batch)
        out["graph_launches"] = per_batch * launches_per_step
    except Exception as e:  # report, do not fail the bench line
        out["graph_us"] = None
        out["graph_error"] = str(e)[:200]
    return out


def run_e2e(args, p, sets, launch, dev, bytes_step, world, dist):
    """Same metric through the C ABI from pinned host buffers: every step uploads its inputs,
    runs, and reads every output back (see pipelined_e2e)."""
    import numpy as np
    import torch

    def pinned(arr):
        if arr is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1).copy())
        return t.pin_memory()

    h_in = {"tokens": pinned(p.tokens), "counts": pinned(p.counts), "scales": pinned(p.scales),
            "topk": pinned(p.topk)}
    if "tokens@0" in sets[0]:
        # multi-source form: each rank's rows go up into that rank's own buffer
        bounds = np.concatenate([[0], np.cumsum(p.counts.astype(np.int64).sum(axis=1))])
        for key, arr, rb in (("tokens", p.tokens, p.row_bytes), ("scales", p.scales, p.scale_row_bytes),
                             ("topk", p.topk, 4)):
            h = h_in.pop(key)
            if arr is not None:
                for i in range(p.N):
                    h_in[f"{key}@{i}"] = h[bounds[i] * rb:bounds[i + 1] * rb]
    outs = ["out_tokens", "out_scales", "out_topk", "idx", "etn"]
    return pipelined_e2e(args, h_in, outs, sets, launch, dev, bytes_step, world, dist)


def pipelined_e2e(args, h_in, outs, sets, launch, dev, bytes_step, world, dist):
    """Every step uploads the pinned host inputs h_in (name -> uint8 tensor) into a device set,
    runs launch(set, stream), and reads the outputs named in outs back to pinned host memory.
    Steps are pipelined over two device buffer sets and three streams (upload / run / read-back,
    ordered by events), so the read-back of step k overlaps the upload of step k+1 on the two
    copy directions."""
    import torch

    two = sets[:2]
    h_out = [{k: (None if s[k] is None else torch.empty(s[k].numel() * s[k].element_size(),
                                                         dtype=torch.uint8).pin_memory())
              for k in outs} for s in two]
    h2d = sum(t.numel() for t in h_in.values() if t is not None)
    d2h = sum(t.numel() for t in h_out[0].values() if t is not None)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_run = torch.cuda.current_stream(dev)
    K = max(3, min(args.steps, 200))
    W = 3
    ev = lambda: torch.cuda.Event()
    up_done = [ev() for _ in range(K + W)]
    run_done = [ev() for _ in range(K + W)]
    down_done = [ev() for _ in range(K + W)]

    def e2e_step(k):
        s, ho = two[k % 2], h_out[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(run_done[k - 2])      # this set's inputs are no longer read
            for name, t in h_in.items():
                if t is not None:
                    s[name].view(torch.uint8).reshape(-1).copy_(t, non_blocking=True)
            up_done[k].record(s_in)
        s_run.wait_event(up_done[k])
        if k >= 2:
            s_run.wait_event(down_done[k - 2])        # this set's outputs were read back
        launch(s, s_run)
        run_done[k].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done[k])
            for name in outs:
                if s[name] is not None:
                    ho[name].copy_(s[name].view(torch.uint8).reshape(-1), non_blocking=True)
            down_done[k].record(s_out)

    for k in range(W):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_run)
    s_in.wait_event(a)
    for k in range(W, W + K):
        e2e_step(k)
    s_run.wait_event(down_done[W + K - 1])
    b.record(s_run)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), dist, dev)
    return {"value": throughput_gbs(world, bytes_step, K, ms), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": ms / K,
            "how": "pinned host buffers; upload, run and read-back on three streams, two device sets"}


# ----------------------------------------------------------------------------- gating top-k

GATING_METRIC = "effective HBM GB/s (read+write) and tokens/sec of MoE gating top-k"


def gating_bytes(w) -> int:
    """x read once, bias read, y (x's dtype) and int32 expert_idx written."""
    T, e = w["x"].shape
    xb = 4 if w["dtype"] == "float32" else 2
    return T * e * xb + (0 if w["bias"] is None else e * xb) + T * w["k"] * (xb + 4)


def gating_oracle_rows(w, rows: int):
    from oracle import gating

    return gating.gating_topk(w["x"][:rows], w["k"], bias=w["bias"], k_group=w["k_group"],
                              group_count=w["group_count"], group_select_mode=w["group_select_mode"],
                              norm_type=w["norm_type"], routed_scaling_factor=w["routed_scaling_factor"],
                              eps=w["eps"])


def gating_config_dict(w, k, extra=None):
    T, e = w["x"].shape
    d = {"workload": w["name"], "op": "gating", "T": T, "e": e, "k": w["k"], "dtype": w["dtype"],
         "group_count": w["group_count"], "k_group": w["k_group"], "norm_type": w["norm_type"],
         "group_select_mode": w["group_select_mode"], "bias": w["bias"] is not None,
         "bytes_per_step": gating_bytes(w)}
    d.update(extra or {})
    return d


def time_gating_oracle(w, budget_s: float, rows: int = 256):
    gating_oracle_rows(w, 8)
    reps, t0 = 0, time.perf_counter()
    while True:
        gating_oracle_rows(w, rows)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    T = w["x"].shape[0]
    return gating_bytes(w) * rows / T * reps / el / 1e9, rows * reps / el, reps, el


def run_gating_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    rows = 64
    for _ in range(args.warmup):
        gating_oracle_rows(w, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        gating_oracle_rows(w, rows)
    el = time.perf_counter() - t0
    T = w["x"].shape[0]
    value = gating_bytes(w) * rows / T * args.steps / el / 1e9
    sample = f"first {rows} of {T} token rows per step"
    print(json.dumps({
        "impl": "reference", "metric": GATING_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": gating_config_dict(w, args.config, {"sample_rows": rows}),
        "tokens_per_s": rows * args.steps / el,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def run_gating(args):
    import numpy as np
    import torch
    import workloads
    from moe_expert_token_gb300 import build as mbuild
    import moe_expert_token_gb300.mrr_v2 as m

    w = workloads.gating_config(args.config)
    if args.impl == "reference":
        return run_gating_reference(args, w)
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        mbuild.build()
    if dist is not None:
        dist.barrier()
    m.load_library()
    tdt = getattr(torch, w["dtype"])
    code = {"float16": m.MRR_GATE_F16, "bfloat16": m.MRR_GATE_BF16, "float32": m.MRR_GATE_F32}[w["dtype"]]
    T, e = w["x"].shape
    k = w["k"]
    B = gating_bytes(w)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, -(-4 * l2 // B))
    x_host = torch.from_numpy(w["x"]).to(tdt)
    bias = None if w["bias"] is None else torch.from_numpy(w["bias"]).to(tdt).to(dev)
    sets = [dict(x=x_host.to(dev), y=torch.empty(T, k, dtype=tdt, device=dev),
                 idx=torch.empty(T, k, dtype=torch.int32, device=dev)) for _ in range(R)]
    ws = torch.empty(4096, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch(s, st):
        r = m.mrr_gating_topk_run(s["x"].data_ptr(), code, T, e, k, None if bias is None else bias.data_ptr(),
                                  None, None, 0, None, None, w["k_group"], w["group_count"],
                                  w["routed_scaling_factor"], w["eps"], w["group_select_mode"], 0,
                                  w["norm_type"], s["y"].data_ptr(), s["idx"].data_ptr(), None,
                                  ws.data_ptr(), ws.numel(), st.cuda_stream)
        if r != m.MRR_OK:
            raise RuntimeError(m.mrr_status_str(r))

    for s in sets:
        launch(s, stream)
    if m.mrr_v2_read_status(ws.data_ptr(), ws.numel(), stream.cuda_stream) != m.MRR_OK:
        raise RuntimeError("gating reported a device error")
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)          # the sampler's first samples; the warm-up follows right before timing
    for i in range(args.warmup):
        launch(sets[i % R], stream)
    K = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.t_start = time.time()
    hold_stream(stream)
    a.record(stream)
    for i in range(K):
        launch(sets[i % R], stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    clocks.t_end = time.time()
    time.sleep(0.2)
    clocks.stop()
    local_ms = a.elapsed_time(b)
    ms = max_over_ranks(local_ms, dist, dev)
    value = throughput_gbs(world, B, K, ms)
    peak, peak_kind = measured_peak()
    achieved = B / (local_ms / K * 1e-3) / 1e9

    # end to end: x uploaded from pinned host memory, y_out and expert_idx read back, every step
    e2e = None
    if not args.no_e2e:
        x_pin = x_host.view(torch.uint8).reshape(-1).pin_memory()
        e2e = pipelined_e2e(args, {"x": x_pin}, ["y", "idx"], sets, launch, dev, B, world, dist)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, tok_s, reps, el = time_gating_oracle(w, min(args.cpu_seconds, 10.0))
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "cpu": cpu_model(), "kind": "oracle",
               "sample": f"the first 256 token rows, {reps} runs in {el:.1f} s, single thread",
               "tokens_per_s": tok_s}
    clock_summary = clocks.summary()
    if rank == 0:
        print(json.dumps({
            "metric": GATING_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy draws shaped like the page's cases)",
            "config": gating_config_dict(w, args.config, {
                "l2": f"{R} rotating buffer sets, {R * B / 1e6:.0f} MB > 4x L2 ({l2 / 1e6:.0f} MB)"}),
            "pct_of_peak": 100.0 * value / world / peak, "tokens_per_s": world * T * K / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": profiled_gating_traffic(args.config),
                         "kernel": "mrr_gate::gating_kernel", "bytes_per_launch": B,
                         "mean_launch_us": local_ms / K * 1e3},
            "issue_roofline": gating_issue_roofline(args.config, local_ms / K * 1e3, clock_summary),
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K, "clocks": clock_summary}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.op == "gating":
        return run_gating(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
