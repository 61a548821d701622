"""GPU parity: the CUDA path against the CPU oracle, element by element, tolerance 0.

The op computes nothing on its payloads (MoeReRoutingV2 article, section 计算公式: rows are
moved, offsets are integer prefixes), so every output must match the oracle bit for bit:
tokens and scales byte-equal, top-k weights equal as 32-bit patterns, index and
expert_token_num equal as integers.  Every call goes through the C ABI.

Coverage: the five workloads at full size (in the launch configuration the benchmark times),
both copy paths, a seeded fuzz sweep over H / dtype width / count type / scale layout / top-k /
idx_type / N*E (across the 4096-segment threshold of the in-kernel scan), plan edits that
stress the bulk pipeline (tiny chunks, many ring wraps, idle CTAs, small and large blocks),
unaligned buffers, the empty problem, identity and transpose cases, and device-detected count
errors.
"""
import functools

import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf, assert_bit_exact, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


@functools.lru_cache(maxsize=2)
def workload(k: int):
    p = workloads.config(k)
    return p, oracle.run_problem(p)


# ------------------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_workload_full_size_default_launch(k):
    p, ref = workload(k)
    gpu = run_gpu(p)
    assert_bit_exact(gpu, ref, p)


@pytest.mark.parametrize("k", [2, 3, 4, 5])
def test_workload_full_size_vector_path(k):
    p, ref = workload(k)
    gpu = run_gpu(p, path=m.MRR_PATH_VECTOR)
    assert_bit_exact(gpu, ref, p)


def test_tiny_workload_both_index_types():
    for it in (0, 1):
        p = workloads.config(1, idx_type=it)
        ref = oracle.run_problem(p)
        for path in (None, m.MRR_PATH_BULK, m.MRR_PATH_VECTOR):
            assert_bit_exact(run_gpu(p, path=path), ref, p)


# ------------------------------------------------------------------------------ fuzz sweep

FUZZ_H = [1, 21, 79, 128, 6057, 7168, 15267, 16383]
DTYPES = ["bfloat16", "int8", "float4_e2m1", "float8_e4m3fn", "float16", "hifloat8",
          "float8_e5m2", "float4_e1m2"]
LAYOUTS = [("none", 0), ("f32_a", 1), ("f32_as", 3), ("e8m0", 8), ("f32_as", 4), ("e8m0", 224)]
NE_SHAPES = [(1, 1), (4, 2), (23, 2), (14, 1), (2, 3), (16, 16), (64, 64), (3, 7), (11, 1),
             (64, 80), (128, 64), (1, 4100), (4097, 1), (8, 32), (32, 8)]


def fuzz_cases(n=64):
    rng = np.random.default_rng(20240)
    cases = []
    for i in range(n):
        N, E = NE_SHAPES[i % len(NE_SHAPES)]
        dt = DTYPES[(i * 3) % len(DTYPES)]
        H = FUZZ_H[(i * 5) % len(FUZZ_H)]
        if workloads.TOKEN_BITS[dt] == 4 and H % 2:
            H -= 1 if H > 1 else -1
        rb = H * workloads.TOKEN_BITS[dt] // 8
        budget = 6 << 20                                   # token bytes per case
        A_max = max(N * E, budget // max(rb, 1))
        if N * E > A_max:                                  # huge N*E: shrink the rows instead
            H = 2 if workloads.TOKEN_BITS[dt] == 4 else 1
        A = int(min(A_max, N * E + rng.integers(0, 3 * N * E + 50)))
        layout, cols = LAYOUTS[i % len(LAYOUTS)]
        cases.append(dict(id=f"{i}-{dt}-H{H}-N{N}E{E}-A{A}-{layout}{cols}", seed=i, A=A, H=H, N=N,
                          E=E, dt=dt, i64=bool(i % 3 == 1), layout=layout, cols=cols,
                          topk=bool(i % 4 != 3), idx=(i // 2) % 2))
    return cases


FUZZ = fuzz_cases()


def fuzz_problem(c):
    rng = np.random.default_rng(7000 + c["seed"])
    return workloads.make_problem(rng, A=c["A"], H=c["H"], N=c["N"], E=c["E"], token_dtype=c["dt"],
                                  count_dtype=np.int64 if c["i64"] else np.int32,
                                  scale_layout=c["layout"], scale_cols=c["cols"],
                                  has_topk=c["topk"], idx_type=c["idx"])


@pytest.mark.parametrize("c", FUZZ, ids=[c["id"] for c in FUZZ])
def test_fuzz(c):
    p = fuzz_problem(c)
    ref = oracle.run_problem(p)
    gpu = run_gpu(p)
    assert_bit_exact(gpu, ref, p)
    assert gpu["plan"]["fuse_scan"] == (1 if c["N"] * c["E"] <= 4096 else 0)
    if gpu["plan"]["path"] == m.MRR_PATH_BULK:
        assert_bit_exact(run_gpu(p, path=m.MRR_PATH_VECTOR), ref, p)


# ------------------------------------------------------------------------------ pipeline stress

STRESS_EDITS = [
    dict(chunk_bytes=16, stages=2, grid=1),            # 1 CTA, thousands of 16-byte chunks
    dict(chunk_bytes=48, stages=3, grid=3),            # ring size not a power of two
    dict(chunk_bytes=4096, stages=8, grid=5, block=64),
    dict(chunk_bytes=65536, stages=2, grid=1022),      # most CTAs own no bytes
    dict(chunk_bytes=1024, stages=5, grid=152, block=1024),
    dict(grid=1, block=64),
    dict(hints=3),
    dict(chunk_bytes=4096, stages=8, hints=1),
    dict(chunk_bytes=8192, stages=3, hints=2),
    dict(sched=0),                                     # equal static slices, no counter
    dict(sched=1, static_chunks=1, chunk_bytes=2048),  # almost everything from the counter
    dict(sched=1, static_chunks=64, chunk_bytes=1024), # static chunks cover the buffer
    dict(sched=1, static_chunks=1, chunk_bytes=16, stages=2, grid=7),
    dict(pdl=0),
    dict(pdl=0, sched=0, grid=300),
    dict(prefetch_chunks=1),                           # L2 prefetch of the next chunks
    dict(prefetch_chunks=64, chunk_bytes=2048, stages=3, grid=9),
    dict(prefetch_chunks=7, sched=0, chunk_bytes=1024),  # static slices: prefetch inside the slice
    dict(prefetch_chunks=40, sched=1, static_chunks=1, chunk_bytes=16, stages=2, grid=7),
]


@pytest.mark.parametrize("edit", STRESS_EDITS, ids=lambda e: "-".join(f"{k}{v}" for k, v in e.items()))
@pytest.mark.parametrize("shape", [(64, 128, 4, 4), (6000, 256, 64, 64), (700, 5000, 8, 32)])
def test_bulk_pipeline_stress(edit, shape):
    A, H, N, E = shape
    p = workloads.make_problem(np.random.default_rng(A + H), A=A, H=H, N=N, E=E,
                               token_dtype="bfloat16", scale_layout="f32_as", scale_cols=4)
    ref = oracle.run_problem(p)
    assert_bit_exact(run_gpu(p, path=m.MRR_PATH_BULK, edit=edit), ref, p)
    vec_edit = {k: v for k, v in edit.items() if k in ("grid", "block", "hints", "sched", "pdl", "prefetch_chunks")}
    assert_bit_exact(run_gpu(p, path=m.MRR_PATH_VECTOR, edit=vec_edit), ref, p)


def test_counter_workspace_reused_across_launches():
    """The chunk counter keeps the previous launch's epoch; every launch must still cover every
    chunk exactly once (garbage at first use, stale values afterwards)."""
    p = workloads.make_problem(np.random.default_rng(77), A=4000, H=2048, N=8, E=16,
                               token_dtype="bfloat16", scale_layout="f32_a", scale_cols=1)
    ref = oracle.run_problem(p)
    ws = DevBuf(1 << 20, "cuda:0", fill=0x5A)
    for k in range(6):
        edit = dict(sched=1, static_chunks=1 + k % 3, chunk_bytes=4096 * (1 + k % 2), grid=16 + 40 * k)
        assert_bit_exact(run_gpu(p, path=m.MRR_PATH_BULK, edit=edit, workspace=ws), ref, p)


# ------------------------------------------------------------------------------ alignment

@pytest.mark.parametrize("offsets", [
    dict(tokens=1), dict(permute_tokens=2), dict(tokens=4, permute_tokens=12),
    dict(tokens=8), dict(scales=2, permute_scales=6), dict(topk=4, permute_topk=8),
    dict(tokens=3, permute_tokens=5, scales=1, permute_scales=3),
])
def test_unaligned_buffers(offsets):
    p = workloads.make_problem(np.random.default_rng(99), A=500, H=300, N=6, E=5,
                               token_dtype="bfloat16", scale_layout="e8m0", scale_cols=10)
    ref = oracle.run_problem(p)
    assert_bit_exact(run_gpu(p, offsets=offsets), ref, p)


def test_forced_bulk_on_unaligned_rows_is_refused():
    p = workloads.make_problem(np.random.default_rng(5), A=40, H=21, N=4, E=2,
                               token_dtype="bfloat16")        # 42-byte rows
    run_gpu(p, path=m.MRR_PATH_BULK, expect_host_status=m.MRR_ERR_PLAN)


# ------------------------------------------------------------------------------ special cases

def test_empty_problem_zero_fills_expert_token_num():
    import torch

    d = torch.device("cuda:0")
    etn = DevBuf(3 * 4, d)
    ws = DevBuf(8192, d)
    st = m.mrr_v2_run(None, m.MRR_BF16, 0, 16, DevBuf(4, d).ptr, 0, 0, 3, None, m.MRR_SCALE_NONE, 0,
                      None, None, None, None, etn.ptr, None, 1, 0, ws.ptr, ws.n,
                      torch.cuda.current_stream().cuda_stream)
    assert st == m.MRR_OK
    assert m.mrr_v2_read_status(ws.ptr, ws.n, torch.cuda.current_stream().cuda_stream) == m.MRR_OK
    assert etn.host().view(np.int32).tolist() == [0, 0, 0]
    assert etn.guards_intact()


@pytest.mark.parametrize("N,E", [(11, 1), (1, 9), (1, 1)])
def test_identity_when_one_rank_or_one_expert(N, E):
    A = 11 if (N, E) == (11, 1) else 50
    p = workloads.make_problem(np.random.default_rng(N * 7 + E), A=A, H=79, N=N, E=E,
                               token_dtype="bfloat16", scale_layout="f32_a", scale_cols=1)
    gpu = run_gpu(p)
    assert np.array_equal(gpu["permute_token_idx"], np.arange(A, dtype=np.int32))
    assert np.array_equal(gpu["permute_tokens"], p.tokens)
    assert_bit_exact(gpu, oracle.run_problem(p), p)


def test_all_ones_counts_is_a_transpose():
    N, E = 16, 16
    c = np.ones((N, E), np.int32)
    p = workloads.make_problem(np.random.default_rng(1), A=N * E, H=7168, N=N, E=E,
                               token_dtype="int8", counts=c)
    gpu = run_gpu(p)
    expect = np.arange(N * E, dtype=np.int32).reshape(N, E).T.ravel()
    assert np.array_equal(gpu["permute_token_idx"], expect)
    assert np.array_equal(gpu["permute_tokens"], p.tokens[expect])


# ------------------------------------------------------------------------------ device-detected errors

@pytest.mark.parametrize("mutate,code", [
    (lambda c: c.__setitem__((0, 1), 0), m.MRR_ERR_COUNT_NONPOS),
    (lambda c: c.__setitem__((1, 0), -5), m.MRR_ERR_COUNT_NONPOS),
    (lambda c: c.__setitem__((2, 2), c[2, 2] + 1), m.MRR_ERR_COUNT_SUM),
    (lambda c: c.__setitem__((2, 2), c[2, 2] - 1) if c[2, 2] > 1 else c.__setitem__((0, 0), c[0, 0] + 1),
     m.MRR_ERR_COUNT_SUM),
])
@pytest.mark.parametrize("big_ne", [False, True])
@pytest.mark.parametrize("path", [m.MRR_PATH_BULK, m.MRR_PATH_VECTOR])
def test_bad_counts_reported_then_recovered(mutate, code, big_ne, path):
    N, E = (80, 64) if big_ne else (4, 4)
    p = workloads.make_problem(np.random.default_rng(3), A=N * E * 3, H=64, N=N, E=E,
                               token_dtype="bfloat16", scale_layout="f32_a", scale_cols=1)
    bad = p.counts.copy()
    mutate(bad)
    ws = DevBuf(1 << 20, "cuda:0")
    out = run_gpu(p, counts=bad, workspace=ws, path=path)
    assert out["status"] == code
    assert out["guards_intact"]
    # the next valid call on the same workspace reports success again
    assert_bit_exact(run_gpu(p, workspace=ws, path=path), oracle.run_problem(p), p)


def test_int64_count_beyond_int32_is_reported():
    p = workloads.make_problem(np.random.default_rng(4), A=64, H=32, N=4, E=4,
                               token_dtype="float16", count_dtype=np.int64)
    bad = p.counts.copy()
    bad[3, 3] = 2**40
    out = run_gpu(p, counts=bad)
    assert out["status"] == m.MRR_ERR_COUNT_SUM


def test_outputs_untouched_when_counts_invalid():
    p = workloads.make_problem(np.random.default_rng(8), A=256, H=128, N=4, E=4,
                               token_dtype="bfloat16")
    bad = p.counts.copy()
    bad[0, 0] = 0
    out = run_gpu(p, counts=bad)
    assert out["status"] == m.MRR_ERR_COUNT_NONPOS
    assert (out["permute_tokens"] == 0xA5).all()
    assert (out["permute_token_idx"].view(np.uint8) == 0xA5).all()


# ------------------------------------------------------------------------------ torch-level call

def test_moe_re_routing_torch_api_matches_oracle():
    import torch

    p = workloads.config(1)
    d = torch.device("cuda:0")
    tok = torch.from_numpy(p.tokens.copy()).view(torch.bfloat16).reshape(p.A, p.H).to(d)
    cnt = torch.from_numpy(p.counts).to(d)
    sc = torch.from_numpy(p.scales.copy()).view(torch.float32).reshape(p.A).to(d)
    tw = torch.from_numpy(p.topk.copy()).reshape(p.A, 1).to(d)
    pt, ps, idx, etn, ptw = m.moe_re_routing(tok, cnt, per_token_scales=sc, expert_topk_weight=tw,
                                             check_status=True)
    ref = oracle.run_problem(p)
    assert np.array_equal(pt.view(torch.uint8).cpu().numpy().reshape(p.A, -1), ref["permute_tokens"])
    assert np.array_equal(ps.view(torch.uint8).cpu().numpy().reshape(p.A, -1), ref["permute_scales"])
    assert np.array_equal(idx.cpu().numpy(), ref["permute_token_idx"])
    assert np.array_equal(etn.cpu().numpy(), ref["expert_token_num"])
    assert np.array_equal(ptw.cpu().numpy().reshape(-1).view(np.uint32),
                          ref["permute_topk_weight"].view(np.uint32))
    # without top-k weights the output is empty (0,); without scales it is an [A] float32
    pt2, ps2, _, _, ptw2 = m.moe_re_routing(tok, cnt)
    assert tuple(ptw2.shape) == (0,) and tuple(ps2.shape) == (p.A,) and ps2.dtype == torch.float32
    assert torch.equal(pt2, pt)


def test_fp8_and_e8m0_torch_dtypes():
    import torch

    p = workloads.make_problem(np.random.default_rng(12), A=300, H=256, N=4, E=8,
                               token_dtype="float8_e4m3fn", scale_layout="e8m0", scale_cols=8)
    d = torch.device("cuda:0")
    tok = torch.from_numpy(p.tokens.copy()).view(torch.float8_e4m3fn).to(d)
    sc = torch.from_numpy(p.scales.copy()).reshape(p.A, 4, 2).to(d)
    tw = torch.from_numpy(p.topk.copy()).reshape(p.A, 1).to(d)
    pt, ps, idx, etn, ptw = m.moe_re_routing(tok, torch.from_numpy(p.counts).to(d),
                                             per_token_scales=sc, expert_topk_weight=tw,
                                             check_status=True)
    ref = oracle.run_problem(p)
    assert np.array_equal(pt.view(torch.uint8).cpu().numpy(), ref["permute_tokens"])
    assert np.array_equal(ps.cpu().numpy().reshape(p.A, -1), ref["permute_scales"])


@pytest.mark.parametrize("bad", [-1, 65])
def test_plan_rejects_prefetch_out_of_range(bad):
    p = workloads.make_problem(np.random.default_rng(5), A=64, H=128, N=4, E=4, token_dtype="bfloat16",
                               scale_layout="none", scale_cols=0)
    run_gpu(p, path=m.MRR_PATH_BULK, edit=dict(prefetch_chunks=bad), expect_host_status=m.MRR_ERR_PLAN)


# ------------------------------------------------------------------------------ many segments

@pytest.mark.parametrize("N,E", [(64, 128), (128, 128), (100, 200), (256, 256)],
                         ids=["8192-staged", "16384-staged", "20000-global-scan", "65536-global"])
@pytest.mark.parametrize("i64", [False, True], ids=["i32", "i64"])
def test_many_segments(N, E, i64):
    """N*E above the fused-scan limit: the scan kernel scans in shared memory up to 16384
    segments (one or two count batches), and the copy kernel stages its tables in shared memory
    while they fit beside the ring; both the forward and the inverse move, bulk and vector paths."""
    from harness import run_gpu_unroute, assert_unroute_bit_exact

    p = workloads.make_problem(np.random.default_rng(N + E + i64), A=2 * N * E + 123, H=64, N=N, E=E,
                               token_dtype="bfloat16", count_dtype=np.int64 if i64 else np.int32,
                               scale_layout="f32_as", scale_cols=2, has_topk=True, idx_type=int(i64))
    ref = oracle.run_problem(p)
    gpu = run_gpu(p)
    assert gpu["plan"]["fuse_scan"] == 0
    assert_bit_exact(gpu, ref, p)
    assert_bit_exact(run_gpu(p, path=m.MRR_PATH_VECTOR), ref, p)
    uref = oracle.unroute(p.tokens, p.counts, permute_scales=p.scales, permute_topk=p.topk)
    assert_unroute_bit_exact(run_gpu_unroute(p), uref, p)
    assert_unroute_bit_exact(run_gpu_unroute(p, path=m.MRR_PATH_VECTOR), uref, p)
    # a smaller ring leaves room to stage the tables of 20000 segments on the bulk path too
    assert_bit_exact(run_gpu(p, path=m.MRR_PATH_BULK, edit=dict(chunk_bytes=16384, stages=2)), ref, p)


# ------------------------------------------------------------------------------ ordering behind a producer

@pytest.mark.parametrize("N,E", [(16, 16), (80, 64), (128, 128)],
                         ids=["fused-scan", "scan-kernel-staged", "scan-kernel-16384"])
def test_inputs_written_by_a_kernel_just_before_the_call(N, E):
    """The kernels run with programmatic stream serialization.  Behind the scan kernel
    (N*E > 4096) the copy kernel starts loading token rows before its own dependency wait: that
    is safe only because the scan kernel waits for its predecessor before it lets the copy kernel
    start.  Here a torch kernel on the same stream writes the tokens and the counts immediately
    before the call, and every output must still match the oracle bit for bit."""
    import torch

    rng = np.random.default_rng(700 + N)
    p = workloads.make_problem(rng, A=max(40000, 3 * N * E), H=1024, N=N, E=E, token_dtype="bfloat16",
                               scale_layout="f32_a", scale_cols=1, has_topk=True)
    ref = oracle.run_problem(p)
    d = torch.device("cuda:0")
    key = 0x5A
    tok_x = torch.from_numpy(p.tokens.reshape(-1) ^ np.uint8(key)).to(d)         # tokens, masked
    cnt_m1 = torch.from_numpy(p.counts.reshape(-1) - 1).to(d)                     # counts - 1
    tok = DevBuf(p.A * p.row_bytes, d)
    cnt = DevBuf(4 * N * E, d)
    sc, tw = DevBuf.of(p.scales, d), DevBuf.of(p.topk, d)
    out_tok, out_sc = DevBuf(p.A * p.row_bytes, d), DevBuf(4 * p.A, d)
    idx, etn, out_tw = DevBuf(4 * p.A, d), DevBuf(4 * E, d), DevBuf(4 * p.A, d)
    st, plan = m.mrr_v2_plan(p.A, p.H, m.MRR_BF16, N, E, 0, m.MRR_SCALE_F32_A, 1, 1, 1, 0, 0)
    assert st == m.MRR_OK and plan.pdl == 1 and plan.fuse_scan == int(N * E <= 4096)
    ws = DevBuf(plan.workspace_bytes, d, fill=0x5A)
    s = torch.cuda.current_stream(d)
    for rep in range(3):
        for b in (tok, cnt, out_tok):                # stale contents the producer must replace
            b.t.fill_(0xA5)
        torch.cuda.synchronize(d)
        # producer kernels, then the op, back to back on one stream with no host sync between
        torch.bitwise_xor(tok_x, key, out=tok.t[tok.off:tok.off + tok.n])
        torch.add(cnt_m1, 1, out=cnt.t[cnt.off:cnt.off + cnt.n].view(torch.int32))
        st = m.mrr_v2_run(tok.ptr, m.MRR_BF16, p.A, p.H, cnt.ptr, 0, N, E, sc.ptr, m.MRR_SCALE_F32_A, 1,
                          tw.ptr, out_tok.ptr, out_sc.ptr, idx.ptr, etn.ptr, out_tw.ptr, 1, 0, ws.ptr, ws.n,
                          s.cuda_stream)
        assert st == m.MRR_OK, m.mrr_status_str(st)
        assert m.mrr_v2_read_status(ws.ptr, ws.n, s.cuda_stream) == m.MRR_OK
        assert np.array_equal(out_tok.host().reshape(p.A, -1), ref["permute_tokens"]), rep
        assert np.array_equal(out_sc.host().reshape(p.A, -1), ref["permute_scales"]), rep
        assert np.array_equal(idx.host().view(np.int32), ref["permute_token_idx"]), rep
        assert np.array_equal(etn.host().view(np.int32), ref["expert_token_num"]), rep
        assert np.array_equal(out_tw.host().view(np.uint32), ref["permute_topk_weight"].view(np.uint32)), rep
        assert all(b.guards_intact() for b in (out_tok, out_sc, idx, etn, out_tw))
