"""GPU parity of the inverse move (expert-major rows back to rank-major order) against the CPU
oracle, bit for bit, through the C ABI (mrr_v2_unroute / mrr_v2_run_plan with direction 1).

The inverse reuses the forward move's segments (MoeReRoutingV2 article, section 计算公式):
tokens[SrcOffset + k] = permute_tokens[DstOffset + k].  Coverage: the five workloads at full
size on both copy paths, a seeded sweep over dtype widths, scale layouts, count types and N*E
(across the 4096-segment threshold), pipeline edits, unaligned buffers, count errors, and the
round trip GPU forward move then GPU inverse, which must give back the input bytes.
"""
import functools

import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf, assert_unroute_bit_exact, run_gpu, run_gpu_unroute

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def unroute_ref(p, counts=None):
    return oracle.unroute(p.tokens, p.counts if counts is None else counts,
                          permute_scales=p.scales, permute_topk=p.topk)


@functools.lru_cache(maxsize=1)
def workload(k: int):
    p = workloads.config(k)
    return p, unroute_ref(p)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("path", [None, m.MRR_PATH_VECTOR])
def test_workload_full_size(k, path):
    p, ref = workload(k)
    assert_unroute_bit_exact(run_gpu_unroute(p, path=path), ref, p)


CASES = [
    # (A, H, N, E, dtype, count dtype, scale layout, cols, topk)
    (64, 128, 4, 4, "bfloat16", np.int32, "f32_a", 1, True),
    (900, 21, 23, 2, "bfloat16", np.int64, "f32_as", 3, True),     # 42-byte rows: vector path
    (700, 6057, 14, 1, "int8", np.int32, "e8m0", 8, False),
    (3000, 79, 11, 1, "float16", np.int32, "none", 0, True),
    (6000, 256, 80, 64, "float8_e4m3fn", np.int64, "e8m0", 224, True),   # 5120 segments
    (9000, 64, 128, 64, "float4_e2m1", np.int32, "f32_a", 1, True),      # 8192 segments
    (2000, 16382, 8, 32, "int8", np.int32, "f32_as", 4, True),
    (4200, 32, 1, 4100, "hifloat8", np.int32, "f32_a", 1, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[4]}-H{c[1]}-N{c[2]}E{c[3]}" for c in CASES])
def test_sweep(case):
    A, H, N, E, dt, cdt, layout, cols, topk = case
    p = workloads.make_problem(np.random.default_rng(A + N), A=A, H=H, N=N, E=E, token_dtype=dt,
                               count_dtype=cdt, scale_layout=layout, scale_cols=cols, has_topk=topk)
    ref = unroute_ref(p)
    gpu = run_gpu_unroute(p)
    assert_unroute_bit_exact(gpu, ref, p)
    assert gpu["plan"]["fuse_scan"] == (1 if N * E <= 4096 else 0)
    if gpu["plan"]["path"] == m.MRR_PATH_BULK:
        assert_unroute_bit_exact(run_gpu_unroute(p, path=m.MRR_PATH_VECTOR), ref, p)


@pytest.mark.parametrize("edit", [
    dict(chunk_bytes=16, stages=2, grid=1),
    dict(sched=0, grid=300),
    dict(sched=1, static_chunks=1, chunk_bytes=2048, grid=37),
    dict(chunk_bytes=4096, stages=8, block=64, pdl=0),
], ids=lambda e: "-".join(f"{k}{v}" for k, v in e.items()))
def test_bulk_pipeline_edits(edit):
    p = workloads.make_problem(np.random.default_rng(5), A=6000, H=256, N=64, E=64,
                               token_dtype="bfloat16", scale_layout="f32_as", scale_cols=4)
    assert_unroute_bit_exact(run_gpu_unroute(p, path=m.MRR_PATH_BULK, edit=edit), unroute_ref(p), p)


@pytest.mark.parametrize("offsets", [dict(permute_tokens=1), dict(tokens=6, scales=2),
                                     dict(permute_tokens=3, tokens=5, permute_scales=1, topk=4)])
def test_unaligned_buffers(offsets):
    p = workloads.make_problem(np.random.default_rng(9), A=500, H=300, N=6, E=5, token_dtype="bfloat16",
                               scale_layout="e8m0", scale_cols=10)
    assert_unroute_bit_exact(run_gpu_unroute(p, offsets=offsets), unroute_ref(p), p)


@pytest.mark.parametrize("k", [3, 5])
def test_round_trip_forward_then_inverse(k):
    """GPU forward move, then the GPU inverse on its outputs: the original bytes come back."""
    p = workloads.config(k)
    fwd = run_gpu(p)
    assert fwd["status"] == m.MRR_OK
    q = workloads.Problem(name=p.name, A=p.A, H=p.H, N=p.N, E=p.E, token_dtype=p.token_dtype,
                          counts=p.counts, tokens=fwd["permute_tokens"], scale_layout=p.scale_layout,
                          scale_cols=p.scale_cols, scales=fwd["permute_scales"],
                          topk=fwd["permute_topk_weight"], idx_type=p.idx_type)
    back = run_gpu_unroute(q)
    assert back["status"] == m.MRR_OK
    assert np.array_equal(back["tokens"], p.tokens)
    if p.scales is not None:
        assert np.array_equal(back["scales"], p.scales)
    if p.topk is not None:
        assert np.array_equal(back["topk_weight"].view(np.uint32), p.topk.view(np.uint32))


@pytest.mark.parametrize("big_ne", [False, True])
def test_bad_counts_reported(big_ne):
    N, E = (80, 64) if big_ne else (4, 4)
    p = workloads.make_problem(np.random.default_rng(13), A=N * E * 2, H=64, N=N, E=E,
                               token_dtype="bfloat16")
    bad = p.counts.copy()
    bad[1, 2] = 0
    out = run_gpu_unroute(p, counts=bad)
    assert out["status"] == m.MRR_ERR_COUNT_NONPOS
    assert (out["tokens"] == 0xA5).all()        # nothing written
    ws = DevBuf(1 << 20, "cuda:0")
    assert run_gpu_unroute(p, counts=bad, workspace=ws)["status"] == m.MRR_ERR_COUNT_NONPOS
    assert_unroute_bit_exact(run_gpu_unroute(p, workspace=ws), unroute_ref(p), p)


def test_unroute_needs_no_index_outputs_and_checks_pairs():
    import torch

    d = torch.device("cuda:0")
    ws = DevBuf(1 << 16, d)
    x = DevBuf(64 * 256, d)
    c = DevBuf.of(np.full((4, 4), 4, np.int32), d)
    s = torch.cuda.current_stream().cuda_stream
    # top-k input without an output
    st = m.mrr_v2_unroute(x.ptr, m.MRR_BF16, 64, 128, c.ptr, 0, 4, 4, None, m.MRR_SCALE_NONE, 0,
                          x.ptr, x.ptr, None, None, ws.ptr, ws.n, s)
    assert st == m.MRR_ERR_TOPK_PAIR
    # the plain move: no index, no per-expert counts anywhere in the call
    y = DevBuf(64 * 256, d)
    st = m.mrr_v2_unroute(x.ptr, m.MRR_BF16, 64, 128, c.ptr, 0, 4, 4, None, m.MRR_SCALE_NONE, 0,
                          None, y.ptr, None, None, ws.ptr, ws.n, s)
    assert st == m.MRR_OK
    assert m.mrr_v2_read_status(ws.ptr, ws.n, s) == m.MRR_OK


def test_torch_level_round_trip():
    import torch

    p = workloads.config(1)
    d = torch.device("cuda:0")
    tok = torch.from_numpy(p.tokens.copy()).view(torch.bfloat16).reshape(p.A, p.H).to(d)
    cnt = torch.from_numpy(p.counts).to(d)
    sc = torch.from_numpy(p.scales.copy()).view(torch.float32).reshape(p.A).to(d)
    tw = torch.from_numpy(p.topk.copy()).reshape(p.A, 1).to(d)
    pt, ps, _, _, ptw = m.moe_re_routing(tok, cnt, per_token_scales=sc, expert_topk_weight=tw,
                                         check_status=True)
    back, bsc, btw = m.moe_re_routing_inverse(pt, cnt, permute_per_token_scales=ps,
                                              permute_topk_weight=ptw, check_status=True)
    assert torch.equal(back.view(torch.int16), tok.view(torch.int16))
    assert torch.equal(bsc.view(torch.int32), sc.view(torch.int32))
    assert torch.equal(btw.view(torch.int32), tw.view(torch.int32))
