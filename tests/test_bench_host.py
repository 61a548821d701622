"""CPU checks of bench.py's host logic: the multi-rank aggregation (max time over ranks, whole-job
throughput) on two gloo ranks, the reference arm's JSON line, the row sampler, and the gating
line's issue roofline."""
import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
    q.put((rank, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_throughput_counts_every_rank():
    # 2 replicas, 1 GB per step each, 10 steps in 1 s -> 20 GB/s for the job
    assert bench.throughput_gbs(2, 10**9, 10, 1000.0) == pytest.approx(20.0)
    assert bench.max_over_ranks(3.5) == 3.5


def test_row_sample_keeps_the_workload_kind():
    p = workloads.config(2)
    q = bench.row_sample(p, 0.05)
    assert q.counts.shape == p.counts.shape and q.counts.dtype == p.counts.dtype
    assert int(q.counts.sum()) == q.A and (q.counts >= 1).all()
    assert q.tokens.shape == (q.A, p.row_bytes)
    # the skew survives: the last cell still holds almost every row
    assert q.counts[-1, -1] == q.A - 255


def test_reference_arm_prints_one_line(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--config", "1", "--steps", "5", "--warmup", "3"]) == 0
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["steps"] == 5 and line["warmup"] == 3


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "5", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_gating_issue_roofline_reads_a_current_summary_only(tmp_path, monkeypatch):
    """The gating line's issue roofline takes the warp instructions per launch from the
    workload's ncu summary only when the summary's source hash is the current one, and divides
    them by the launch time against SMs x 4 schedulers x the sampled SM clock."""
    (tmp_path / "profiles").mkdir()
    name = bench.GATING_PROFILES[2]
    (tmp_path / "profiles" / name).write_text(
        "kernel_source_sha256: 0123abcd\ntraffic_bytes_per_launch: 1000\n"
        "warp_instructions_per_launch: 7000000\n", encoding="utf-8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "gating_source_hash", lambda: "0123abcd")
    assert bench.profiled_gating_traffic(2) == 1000
    r = bench.gating_issue_roofline(2, 10.0, {"sm_mhz": 2000.0})
    assert r["bound"] == "issue" and r["warp_instructions_per_launch"] == 7000000
    assert r["peak"] == pytest.approx(152 * 4 * 2000e6)
    assert r["achieved"] == pytest.approx(7e6 / 10e-6)
    assert r["frac"] == pytest.approx(7e11 / (152 * 4 * 2e9))
    assert bench.gating_issue_roofline(2, 10.0, {"sm_mhz": None})["sm_mhz"] == 2070.0
    assert bench.gating_issue_roofline(1, 10.0, {}) is None          # no summary for workload 1 here
    monkeypatch.setattr(bench, "gating_source_hash", lambda: "ffff0000")
    assert bench.gating_issue_roofline(2, 10.0, {"sm_mhz": 2000.0}) is None
    assert bench.profiled_gating_traffic(2) is None
