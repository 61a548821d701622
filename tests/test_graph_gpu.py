"""Launches captured in a CUDA graph and replayed.

A replayed launch keeps the parameters it was captured with, including the host's launch epoch.
The chunk counter is returned to 0 by the launch that draws its last value, so each replay must
still move every chunk exactly once: the outputs are poisoned before every replay and must come
out bit-exact.  The dynamic scheduler is forced with many small chunks, a first ticket claimed by
every CTA, and two workspaces shared by three captured launches.
"""
import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf, assert_bit_exact, ptr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def _buffers(p, d):
    c = p.counts
    return dict(tok=DevBuf.of(p.tokens, d), cnt=DevBuf.of(c, d), sc=DevBuf.of(p.scales, d),
                tw=DevBuf.of(p.topk, d), out_tok=DevBuf(p.A * p.row_bytes, d),
                out_sc=DevBuf(p.A * p.scale_row_bytes, d), idx=DevBuf(4 * p.A, d),
                etn=DevBuf(p.E * c.dtype.itemsize, d), out_tw=DevBuf(4 * p.A, d))


def _poison(b):
    for key in ("out_tok", "out_sc", "idx", "etn", "out_tw"):
        b[key].t[b[key].off:b[key].off + b[key].n].fill_(0xEE)


def _result(b, p):
    return {"status": m.MRR_OK,
            "permute_tokens": b["out_tok"].host().reshape(p.A, p.row_bytes),
            "permute_scales": b["out_sc"].host().reshape(p.A, p.scale_row_bytes),
            "permute_token_idx": b["idx"].host().view(np.int32),
            "expert_token_num": b["etn"].host().view(p.counts.dtype),
            "permute_topk_weight": b["out_tw"].host().view(np.float32),
            "guards_intact": all(b[k].guards_intact() for k in ("out_tok", "out_sc", "idx", "etn", "out_tw")),
            "inputs_intact": np.array_equal(b["tok"].host(), np.ascontiguousarray(p.tokens).reshape(-1))}


@pytest.mark.parametrize("edit", [dict(sched=1, static_chunks=1, chunk_bytes=16384, grid=16),
                                  dict(sched=1, static_chunks=1, chunk_bytes=4096, stages=4, grid=64)])
def test_graph_replays_move_every_chunk(edit):
    import torch

    p = workloads.make_problem(np.random.default_rng(99), A=4000, H=2048, N=8, E=16,
                               token_dtype="bfloat16", scale_layout="f32_a", scale_cols=1)
    ref = oracle.run_problem(p)
    d = torch.device("cuda:0")
    code, sl = m.DTYPE_CODES[p.token_dtype], m.SCALE_CODES[p.scale_layout]
    st, plan = m.mrr_v2_plan(p.A, p.H, code, p.N, p.E, 0, sl, p.scale_cols, 1, 1, p.idx_type, 0)
    assert st == m.MRR_OK
    plan.path = m.MRR_PATH_BULK
    for k, v in edit.items():
        setattr(plan, k, v)
    sets = [_buffers(p, d) for _ in range(2)]
    wss = [DevBuf(1 << 20, d, fill=0x5A) for _ in range(2)]

    def launch(b, ws, stream):
        st = m.mrr_v2_run_plan(plan, ptr(b["tok"]), code, ptr(b["cnt"]), ptr(b["sc"]), ptr(b["tw"]),
                               ptr(b["out_tok"]), ptr(b["out_sc"]), ptr(b["idx"]), ptr(b["etn"]),
                               ptr(b["out_tw"]), p.expert_token_num_type, ws.ptr, ws.n, stream)
        assert st == m.MRR_OK, m.mrr_status_str(st)

    # one eager launch per set first, so the counters already hold tags of earlier launches
    for b, ws in zip(sets, wss):
        launch(b, ws, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        for i in range(3):   # set 0, set 1, set 0 again: two launches per replay on workspace 0
            launch(sets[i % 2], wss[i % 2], cap.cuda_stream)
    for _ in range(3):
        for b in sets:
            _poison(b)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for b, ws in zip(sets, wss):
            assert m.mrr_v2_read_status(ws.ptr, ws.n, torch.cuda.current_stream().cuda_stream) == m.MRR_OK
            assert_bit_exact(_result(b, p), ref, p)


def test_graph_replays_gating():
    """The gating op carries no cross-launch state; replays must match an eager launch."""
    import torch

    rng = np.random.default_rng(7)
    T, e, k = 512, 256, 8
    x = torch.from_numpy(rng.standard_normal((T, e)).astype(np.float32)).to(torch.bfloat16).cuda()
    bias = torch.from_numpy((rng.random(e) * 0.1).astype(np.float32)).to(torch.bfloat16).cuda()
    kw = dict(bias=bias, k_group=4, group_count=8, group_select_mode=1, norm_type=1,
              routed_scaling_factor=2.5, eps=1e-20)
    y_ref, i_ref, _ = m.moe_gating_top_k(x, k, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        y, idx, _ = m.moe_gating_top_k(x, k, **kw)
    for _ in range(2):
        y.fill_(0)
        idx.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(idx, i_ref) and torch.equal(y, y_ref)


def test_concurrent_streams_with_their_own_workspaces():
    """Launches on two streams at once, each with its own workspace (as the header requires), both
    through the dynamic scheduler: every output bit-exact, four rounds."""
    import torch

    p = workloads.make_problem(np.random.default_rng(123), A=6000, H=2048, N=8, E=16,
                               token_dtype="bfloat16", scale_layout="f32_a", scale_cols=1)
    ref = oracle.run_problem(p)
    d = torch.device("cuda:0")
    code, sl = m.DTYPE_CODES[p.token_dtype], m.SCALE_CODES[p.scale_layout]
    st, plan = m.mrr_v2_plan(p.A, p.H, code, p.N, p.E, 0, sl, p.scale_cols, 1, 1, p.idx_type, 0)
    assert st == m.MRR_OK
    plan.path = m.MRR_PATH_BULK
    plan.sched, plan.static_chunks, plan.chunk_bytes, plan.grid = 1, 1, 16384, 48
    sets = [_buffers(p, d) for _ in range(2)]
    wss = [DevBuf(1 << 20, d, fill=0x5A) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(4):
        for b in sets:
            _poison(b)
        torch.cuda.synchronize()
        for b, ws, s in zip(sets, wss, streams):
            st = m.mrr_v2_run_plan(plan, ptr(b["tok"]), code, ptr(b["cnt"]), ptr(b["sc"]), ptr(b["tw"]),
                                   ptr(b["out_tok"]), ptr(b["out_sc"]), ptr(b["idx"]), ptr(b["etn"]),
                                   ptr(b["out_tw"]), p.expert_token_num_type, ws.ptr, ws.n, s.cuda_stream)
            assert st == m.MRR_OK
        torch.cuda.synchronize()
        for b, ws in zip(sets, wss):
            assert m.mrr_v2_read_status(ws.ptr, ws.n, torch.cuda.current_stream().cuda_stream) == m.MRR_OK
            assert_bit_exact(_result(b, p), ref, p)


@pytest.mark.parametrize("N,E", [(8, 16), (70, 64)], ids=["fused-scan", "scan-kernel"])
def test_graph_replays_multi_source(N, E):
    """The multi-source form captured in a CUDA graph: its pointer tables live in device memory, so
    a replay reads whatever rows the per-rank buffers hold at that moment.  The buffers are
    rewritten with new rows between replays, and every replay must match the oracle on them."""
    import torch

    d = torch.device("cuda:0")
    A, H = 3 * N * E + 500, 1024
    base = workloads.make_problem(np.random.default_rng(300 + N), A=A, H=H, N=N, E=E, token_dtype="bfloat16",
                                  scale_layout="f32_as", scale_cols=2, has_topk=True)
    bounds = np.concatenate([[0], np.cumsum(base.counts.astype(np.int64).sum(axis=1))])
    rb, sb = base.row_bytes, base.scale_row_bytes
    tok = [DevBuf(int(bounds[i + 1] - bounds[i]) * rb, d) for i in range(N)]
    sc = [DevBuf(int(bounds[i + 1] - bounds[i]) * sb, d) for i in range(N)]
    tw = [DevBuf(int(bounds[i + 1] - bounds[i]) * 4, d) for i in range(N)]
    tab = {k: torch.tensor([b.ptr for b in v], dtype=torch.int64, device=d) for k, v in
           (("tok", tok), ("sc", sc), ("tw", tw))}
    rows = torch.tensor(np.diff(bounds), dtype=torch.int64, device=d)
    cnt = DevBuf.of(base.counts, d)
    outs = dict(out_tok=DevBuf(A * rb, d), out_sc=DevBuf(A * sb, d), idx=DevBuf(4 * A, d),
                etn=DevBuf(E * 4, d), out_tw=DevBuf(4 * A, d))
    st, plan = m.mrr_v2_plan(A, H, m.MRR_BF16, N, E, 0, m.MRR_SCALE_F32_AS, 2, 1, 1, 0, 0)
    assert st == m.MRR_OK
    ws = DevBuf(plan.workspace_bytes, d, fill=0x5A)

    def fill(p):   # the problem's rows into the per-rank buffers
        for i in range(N):
            for bl, arr, w in ((tok, p.tokens, rb), (sc, p.scales, sb), (tw, p.topk.view(np.uint8).reshape(A, 4), 4)):
                part = np.ascontiguousarray(arr).reshape(A, w)[bounds[i]:bounds[i + 1]].reshape(-1)
                bl[i].t[bl[i].off:bl[i].off + bl[i].n].copy_(torch.from_numpy(part.copy()).to(d))

    def launch(stream):
        st = m.mrr_v2_run_multi(tab["tok"].data_ptr(), tab["sc"].data_ptr(), tab["tw"].data_ptr(), rows.data_ptr(),
                                m.MRR_BF16, A, H, cnt.ptr, 0, N, E, m.MRR_SCALE_F32_AS, 2, outs["out_tok"].ptr,
                                outs["out_sc"].ptr, outs["idx"].ptr, outs["etn"].ptr, outs["out_tw"].ptr, 1, 0,
                                ws.ptr, ws.n, stream)
        assert st == m.MRR_OK, m.mrr_status_str(st)

    fill(base)
    launch(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        launch(cap.cuda_stream)
    for rep in range(3):
        p = workloads.make_problem(np.random.default_rng(400 + rep), A=A, H=H, N=N, E=E, token_dtype="bfloat16",
                                   counts=base.counts, scale_layout="f32_as", scale_cols=2, has_topk=True)
        fill(p)
        _poison(outs)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert m.mrr_v2_read_status(ws.ptr, ws.n, torch.cuda.current_stream().cuda_stream) == m.MRR_OK
        ref = oracle.run_problem(p)
        got = {"status": m.MRR_OK,
               "permute_tokens": outs["out_tok"].host().reshape(A, rb),
               "permute_scales": outs["out_sc"].host().reshape(A, sb),
               "permute_token_idx": outs["idx"].host().view(np.int32),
               "expert_token_num": outs["etn"].host().view(np.int32),
               "permute_topk_weight": outs["out_tw"].host().view(np.float32),
               "guards_intact": all(b.guards_intact() for b in outs.values()), "inputs_intact": True}
        assert_bit_exact(got, ref, p)
