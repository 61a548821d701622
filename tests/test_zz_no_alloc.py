"""mrr_v2_run_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace.  Examples are a framework plugin that receives
only its input and output tensors, a server whose device memory budget is fixed at start-up, and
code that must avoid cudaMalloc/cudaFree because those calls can synchronise the device.  For
them, mrr_v2_run_noalloc uses a fixed array in the library's own device memory as scratch.

This test calls it through the C ABI twice in a row, on two different problems.  Both problems
have more than 4096 segments, so the shared scratch holds the offset tables.  It compares every
output, bit for bit, with what mrr_v2_run produces from its own workspace, and with the CPU
oracle.  Further cases run at the segment limit (N*E = 16384, both offset tables filling the
array) and below 4096 segments (only the status words and the chunk counter live in the array);
it also checks that larger problems are refused, and the optional wait-and-check readback.

The file is named so that pytest collects it last.  It builds and loads everything it needs
itself, so it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()
    return torch.device("cuda:0")


def _buffers(p, dev):
    import torch

    def up(a):
        if a is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1).copy()).to(dev)

    ins = dict(tok=up(p.tokens), cnt=up(p.counts), sc=up(p.scales), tw=up(p.topk))

    def outs():
        return dict(
            tok=torch.full((p.A * p.row_bytes,), 0x11, dtype=torch.uint8, device=dev),
            sc=None if p.scales is None else torch.full((p.A * p.scale_row_bytes,), 0x22,
                                                        dtype=torch.uint8, device=dev),
            idx=torch.full((p.A,), -1, dtype=torch.int32, device=dev),
            etn=torch.full((p.E * p.counts.dtype.itemsize,), 0x33, dtype=torch.uint8, device=dev),
            tw=None if p.topk is None else torch.full((4 * p.A,), 0x44, dtype=torch.uint8, device=dev))
    return ins, outs


def _p(t):
    return None if t is None else t.data_ptr()


def _run_existing(p, ins, o, dev):
    import torch

    st, plan = m.mrr_v2_plan(p.A, p.H, m.DTYPE_CODES[p.token_dtype], p.N, p.E, p.count_is_i64,
                             m.SCALE_CODES[p.scale_layout], p.scale_cols, p.topk is not None, 1,
                             p.idx_type, 0)
    assert st == m.MRR_OK
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    st = m.mrr_v2_run(_p(ins["tok"]), m.DTYPE_CODES[p.token_dtype], p.A, p.H, _p(ins["cnt"]),
                      p.count_is_i64, p.N, p.E, _p(ins["sc"]), m.SCALE_CODES[p.scale_layout],
                      p.scale_cols, _p(ins["tw"]), _p(o["tok"]), _p(o["sc"]), _p(o["idx"]),
                      _p(o["etn"]), _p(o["tw"]), 1, p.idx_type, ws.data_ptr(), ws.numel(), s)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    assert m.mrr_v2_read_status(ws.data_ptr(), ws.numel(), s) == m.MRR_OK


def _run_noalloc(p, ins, o, dev, wait_and_check=1, counts=None):
    import torch

    s = torch.cuda.current_stream(dev).cuda_stream
    return m.mrr_v2_run_noalloc(_p(ins["tok"]), m.DTYPE_CODES[p.token_dtype], p.A, p.H,
                                _p(counts if counts is not None else ins["cnt"]), p.count_is_i64,
                                p.N, p.E, _p(ins["sc"]), m.SCALE_CODES[p.scale_layout],
                                p.scale_cols, _p(ins["tw"]), _p(o["tok"]), _p(o["sc"]),
                                _p(o["idx"]), _p(o["etn"]), _p(o["tw"]), 1, p.idx_type,
                                wait_and_check, s)


def _same(a, b):
    for k in a:
        if a[k] is None:
            assert b[k] is None
            continue
        assert a[k].dtype == b[k].dtype and a[k].shape == b[k].shape, k
        assert bool((a[k] == b[k]).all().item()), f"{k} differs from mrr_v2_run's output"


def _matches_oracle(p, o):
    """Every output of one call equal to the CPU oracle's, bit for bit."""
    ref = oracle.run_problem(p)
    assert np.array_equal(o["tok"].cpu().numpy().reshape(p.A, -1), ref["permute_tokens"])
    assert np.array_equal(o["idx"].cpu().numpy(), ref["permute_token_idx"])
    assert np.array_equal(o["etn"].cpu().numpy().view(p.counts.dtype), ref["expert_token_num"])
    if p.scales is not None:
        assert np.array_equal(o["sc"].cpu().numpy().reshape(p.A, -1), ref["permute_scales"])
    if p.topk is not None:
        assert np.array_equal(o["tw"].cpu().numpy().view(np.uint32),
                              ref["permute_topk_weight"].view(np.uint32))


def _compare_both(p, dev):
    import torch

    ins, outs = _buffers(p, dev)
    ref, got = outs(), outs()
    _run_existing(p, ins, ref, dev)
    st = _run_noalloc(p, ins, got, dev)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    torch.cuda.synchronize(dev)
    _same(ref, got)
    _matches_oracle(p, got)


def test_noalloc_matches_mrr_v2_run_on_two_calls_in_a_row(dev):
    import torch

    problems = [
        workloads.make_problem(np.random.default_rng(61), A=30000, H=512, N=80, E=64,
                               token_dtype="bfloat16", count_dtype=np.int32,
                               scale_layout="f32_as", scale_cols=4, has_topk=True, idx_type=0),
        workloads.make_problem(np.random.default_rng(62), A=20000, H=300, N=70, E=90,
                               token_dtype="int8", count_dtype=np.int64,
                               scale_layout="e8m0", scale_cols=10, has_topk=True, idx_type=1),
    ]
    for p in problems:
        assert p.N * p.E > 4096      # the offset tables live in the shared scratch
        _compare_both(p, dev)


def test_noalloc_at_the_segment_limit_and_below_the_fused_limit(dev):
    """N*E = 16384 exactly (the bulk path; both tables fill the array), then N*E = 256 (each CTA
    scans the counts itself; only the status words and the chunk counter are in the array), then
    the limit case once more on the array the small call left behind."""
    limit = workloads.make_problem(np.random.default_rng(65), A=40000, H=256, N=128, E=128,
                                   token_dtype="bfloat16", count_dtype=np.int32,
                                   scale_layout="f32_a", scale_cols=1, has_topk=True, idx_type=0)
    assert limit.N * limit.E == m.MRR_NOALLOC_MAX_SEGMENTS
    small = workloads.make_problem(np.random.default_rng(66), A=50000, H=2048, N=16, E=16,
                                   token_dtype="int8", count_dtype=np.int64,
                                   scale_layout="f32_as", scale_cols=3, has_topk=True, idx_type=1)
    for p in (limit, small, limit):
        _compare_both(p, dev)


def test_noalloc_rejects_too_many_segments(dev):
    p = workloads.make_problem(np.random.default_rng(63), A=16385 * 2, H=8, N=16385, E=1,
                               token_dtype="int8", scale_layout="none", scale_cols=0,
                               has_topk=False)
    ins, outs = _buffers(p, dev)
    o = outs()
    assert _run_noalloc(p, ins, o, dev) == m.MRR_ERR_WORKSPACE
    assert bool((o["idx"] == -1).all().item())          # nothing was enqueued


def test_noalloc_reports_bad_counts_then_recovers(dev):
    import torch

    p = workloads.make_problem(np.random.default_rng(64), A=9000, H=64, N=40, E=128,
                               token_dtype="float16", scale_layout="f32_a", scale_cols=1)
    ins, outs = _buffers(p, dev)
    bad = p.counts.copy()
    bad[3, 5] = 0
    bad_dev = torch.from_numpy(bad).to(dev)
    assert _run_noalloc(p, ins, outs(), dev, counts=bad_dev) == m.MRR_ERR_COUNT_NONPOS
    ref, got = outs(), outs()
    _run_existing(p, ins, ref, dev)
    assert _run_noalloc(p, ins, got, dev) == m.MRR_OK
    torch.cuda.synchronize(dev)
    _same(ref, got)
