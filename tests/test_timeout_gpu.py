"""The copy kernel's bounded-wait error path, driven to its end without hanging anything.

The bulk path hands out chunks from a counter in the workspace, tagged with the launch's epoch.
A ticket larger than any this launch can draw means the counter was left by a run that never
finished its claims; the kernel must then flag MRR_ERR_TIMEOUT and leave at once (no wait, no
trap).  Here the host plants such a counter: the plan fixes the launch's epoch (plan.epoch) and
the workspace's counter word (bytes 4096..4103) is written as (epoch << 24) | 2^23, a ticket far
above the launch's last one.  Every CTA that reaches the dynamic chunks draws a ticket from
there and stops.  The call must report MRR_ERR_TIMEOUT promptly with every guard band intact,
and the next call on a zeroed counter must be bit-exact against the oracle.

This mirrors the host-side rejection of bad inputs that the "CANN ops-transformer
MoeReRoutingV2" article describes (section 参数取值细节): an error is reported, not a hang.
"""
import time

import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf, assert_bit_exact, run_gpu

pytestmark = pytest.mark.gpu

TICKET_OFFSET = 4096     # the chunk counter's byte offset in the workspace


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def _plant_counter(ws: DevBuf, value: int):
    import torch

    raw = np.array([value], dtype=np.uint64).view(np.uint8)
    ws.t[ws.off + TICKET_OFFSET:ws.off + TICKET_OFFSET + 8].copy_(torch.from_numpy(raw.copy()).to(ws.t.device))


@pytest.mark.parametrize("N,E", [(16, 16), (64, 80)])    # fused scan, and the scan kernel ahead
def test_planted_stale_counter_reports_timeout_then_recovers(N, E):
    import torch

    rng = np.random.default_rng(900 + N)
    p = workloads.make_problem(rng, A=8192, H=2048, N=N, E=E, token_dtype="bfloat16",
                               scale_layout="f32_a", scale_cols=1, has_topk=True)
    st, plan = m.mrr_v2_plan(p.A, p.H, m.DTYPE_CODES[p.token_dtype], N, E, 0, m.MRR_SCALE_F32_A, 1, 1, 1,
                             p.idx_type, 0)
    assert st == m.MRR_OK and plan.path == m.MRR_PATH_BULK and plan.sched == 1
    epoch = 0x5A5A5A5A5
    # one static chunk per CTA, so most chunks are served by the counter
    edit = {"sched": 1, "static_chunks": 1, "epoch": epoch}
    ws = DevBuf(plan.workspace_bytes, torch.device("cuda:0"), 0, fill=0x5A)

    _plant_counter(ws, (epoch << 24) | (1 << 23))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bad = run_gpu(p, edit=edit, workspace=ws)
    elapsed = time.perf_counter() - t0
    assert bad["status"] == m.MRR_ERR_TIMEOUT, m.mrr_status_str(bad["status"])
    assert bad["guards_intact"]
    assert elapsed < 1.0, f"the kernel took {elapsed:.2f} s to give up: it must not wait"

    # a zeroed counter (the documented recovery), the same fixed epoch: every row moves
    _plant_counter(ws, 0)
    good = run_gpu(p, edit=edit, workspace=ws)
    assert_bit_exact(good, oracle.run_problem(p), p)
    # and again without touching the counter: the finished run's count is recognised
    again = run_gpu(p, edit=edit, workspace=ws)
    assert_bit_exact(again, oracle.run_problem(p), p)


def test_plan_rejects_epoch_out_of_range():
    import torch

    p = workloads.config(1)
    for bad in (-1, 1 << 40):
        out = run_gpu(p, edit={"epoch": bad}, expect_host_status=m.MRR_ERR_PLAN)
        assert out["host_status"] == m.MRR_ERR_PLAN
    torch.cuda.synchronize()
