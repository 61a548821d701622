"""GPU parity of the multi-source form (mrr_v2_run_multi / mrr_v2_run_plan_multi) against the oracle.

The dispatch ("torch_npu.npu_moe_distribute_dispatch" page: expand_x, ep_recv_counts) delivers
each peer's rows; the re-routing ("CANN ops-transformer MoeReRoutingV2" article, sections 计算公式
and 数据流定位) lays them out expert-major.  In the multi-source form rank i's rows stay in a
buffer of their own (a separate allocation, or a fixed-capacity slot of one receive buffer), and
the op reads them there.  Its outputs must equal, bit for bit, the oracle run on the
concatenation of the N buffers in rank order: the rank-major input of the single-source op.

Coverage: the large workloads at full size on both copy paths, a seeded fuzz over H, dtype width,
count type, scale layout, top-k, idx_type and N*E (across the 4096-segment threshold and the
staged / global table limits), both source layouts, sources at odd byte offsets (vector path),
and the device-side refusals: a NULL pointer, a token source that is not 16-byte aligned on the
bulk path, and counts that exceed a rank's capacity, each followed by a valid call.
"""
import functools

import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf, assert_bit_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def rank_rows(counts: np.ndarray) -> np.ndarray:
    """Row boundaries of the ranks in the rank-major order: [0, r0, r0 + r1, ..., A]."""
    return np.concatenate([[0], np.cumsum(counts.astype(np.int64).sum(axis=1))])


def run_gpu_multi(p, *, layout="separate", path=None, edit=None, src_offset=0, sc_offset=0, tk_offset=0,
                  spare_rows=0, rows_given=True, rows_override=None, null_rank=None, counts=None,
                  workspace=None, device="cuda:0", expect_host_status=m.MRR_OK):
    """Run the multi-source form on problem ``p``: rank i's token / scale / top-k rows are cut
    out of the problem's rank-major arrays and placed in per-rank buffers.

    layout "separate": one guard-banded buffer per rank and array, starting ``*_offset`` bytes
    past an aligned address; "slots": one buffer per array holding N slots of
    (rows_i + spare_rows) rows each (the capacity passed in src_rows).  ``null_rank`` puts NULL
    in the token table for that rank."""
    import torch

    d = torch.device(device)
    c = p.counts if counts is None else counts
    N, E = c.shape
    bounds = rank_rows(p.counts)
    rows = np.diff(bounds)
    code, sl = m.DTYPE_CODES[p.token_dtype], m.SCALE_CODES[p.scale_layout]
    arrays = {"tok": (p.tokens, p.row_bytes, src_offset),
              "sc": (p.scales, p.scale_row_bytes, sc_offset),
              "tk": (None if p.topk is None else p.topk.view(np.uint8).reshape(p.A, 4), 4, tk_offset)}
    bufs, tables, cap = {}, {}, rows + spare_rows
    for key, (arr, rb, off) in arrays.items():
        if arr is None:
            tables[key] = None
            continue
        raw = np.ascontiguousarray(arr).reshape(p.A, rb)
        if layout == "separate":
            bl = [DevBuf.of(raw[bounds[i]:bounds[i + 1]], d, offset=off) for i in range(N)]
            ptrs = [b.ptr for b in bl]
        else:
            slot = np.full((N, int(cap.max()), rb), 0xC3, np.uint8)
            for i in range(N):
                slot[i, :rows[i]] = raw[bounds[i]:bounds[i + 1]]
            bl = [DevBuf.of(slot, d, offset=off)]
            ptrs = [bl[0].ptr + i * int(cap.max()) * rb for i in range(N)]
        if key == "tok" and null_rank is not None:
            ptrs[null_rank] = 0
        bufs[key] = bl
        tables[key] = torch.tensor(ptrs, dtype=torch.int64, device=d)
    if layout == "slots":
        cap = np.full(N, int(cap.max()))
    src_rows = None
    if rows_given:
        src_rows = torch.tensor(cap if rows_override is None else rows_override, dtype=torch.int64, device=d)
    cnt = DevBuf.of(c, d)
    out_tok = DevBuf(p.A * p.row_bytes, d)
    out_sc = None if p.scales is None else DevBuf(p.A * p.scale_row_bytes, d)
    idx = DevBuf(4 * p.A, d)
    etn = DevBuf(E * c.dtype.itemsize, d)
    out_tw = None if p.topk is None else DevBuf(4 * p.A, d)
    st, plan = m.mrr_v2_plan(p.A, p.H, code, N, E, c.dtype == np.int64, sl, p.scale_cols, p.topk is not None,
                             p.expert_token_num_type, p.idx_type, d.index or 0)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    if workspace is None:
        workspace = DevBuf(plan.workspace_bytes, d, fill=0x5A)
    ins = [b for bl in bufs.values() for b in bl]
    copies = [b.t.clone() for b in ins]
    P = lambda x: None if x is None else (x.ptr if isinstance(x, DevBuf) else x.data_ptr())
    stream = torch.cuda.current_stream(d).cuda_stream
    if path is None and not edit:
        st = m.mrr_v2_run_multi(P(tables["tok"]), P(tables["sc"]), P(tables["tk"]), P(src_rows), code, p.A, p.H,
                                P(cnt), c.dtype == np.int64, N, E, sl, p.scale_cols, P(out_tok), P(out_sc), P(idx),
                                P(etn), P(out_tw), p.expert_token_num_type, p.idx_type, workspace.ptr, workspace.n,
                                stream)
    else:
        if path is not None:
            plan.path = path
        for k, v in (edit or {}).items():
            setattr(plan, k, v)
        st = m.mrr_v2_run_plan_multi(plan, P(tables["tok"]), P(tables["sc"]), P(tables["tk"]), P(src_rows), code,
                                     P(cnt), P(out_tok), P(out_sc), P(idx), P(etn), P(out_tw),
                                     p.expert_token_num_type, workspace.ptr, workspace.n, stream)
    assert st == expect_host_status, m.mrr_status_str(st)
    out = {"host_status": st, "plan": plan.as_dict()}
    if st != m.MRR_OK:
        return out
    out["status"] = m.mrr_v2_read_status(workspace.ptr, workspace.n, stream)
    torch.cuda.synchronize(d)
    out["permute_tokens"] = out_tok.host().reshape(p.A, p.row_bytes)
    out["permute_scales"] = None if out_sc is None else out_sc.host().reshape(p.A, p.scale_row_bytes)
    out["permute_token_idx"] = idx.host().view(np.int32)
    out["expert_token_num"] = etn.host().view(c.dtype)
    out["permute_topk_weight"] = None if out_tw is None else out_tw.host().view(np.float32)
    out["guards_intact"] = all(b.guards_intact() for b in (out_tok, out_sc, idx, etn, out_tw) if b is not None)
    out["inputs_intact"] = all(torch.equal(b.t, c0) for b, c0 in zip(ins, copies))
    return out


@functools.lru_cache(maxsize=2)
def workload(k: int):
    p = workloads.config(k)
    return p, oracle.run_problem(p)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_workload_full_size(k):
    p, ref = workload(k)
    assert_bit_exact(run_gpu_multi(p), ref, p)


@pytest.mark.parametrize("k", [2, 4])
def test_workload_full_size_vector_path(k):
    p, ref = workload(k)
    assert_bit_exact(run_gpu_multi(p, path=m.MRR_PATH_VECTOR), ref, p)


@pytest.mark.parametrize("k", [4, 5])      # ranks of similar size: the slots stay small
def test_workload_full_size_receive_slots(k):
    p, ref = workload(k)
    assert_bit_exact(run_gpu_multi(p, layout="slots", spare_rows=37), ref, p)


FUZZ = []
_rng = np.random.default_rng(4242)
_dtypes = list(m.DTYPE_CODES)
_H = [1, 21, 79, 128, 6057, 7168, 15267, 16383]
_NE = [(1, 1), (1, 5), (7, 1), (4, 4), (3, 50), (16, 16), (64, 64), (80, 64), (100, 200)]
for _c in range(28):
    dt = _dtypes[_c % len(_dtypes)]
    H = int(_H[_rng.integers(len(_H))])
    if dt.startswith("float4") and H % 2:
        H -= 1 if H > 1 else -1
    N, E = _NE[_c % len(_NE)]
    FUZZ.append(dict(case=_c, dt=dt, H=H, N=N, E=E, i64=bool(_c % 3 == 0),
                     sl=["none", "f32_a", "f32_as", "e8m0"][_c % 4], topk=bool(_c % 2),
                     idx=int(_c % 5 == 0), layout=["separate", "slots"][(_c // 2) % 2],
                     off=int(_rng.integers(0, 16)) if _c % 4 == 1 else 0))


@pytest.mark.parametrize("c", FUZZ, ids=lambda c: f"case{c['case']}-{c['dt']}-H{c['H']}-{c['N']}x{c['E']}")
def test_fuzz(c):
    rng = np.random.default_rng(5000 + c["case"])
    NE = c["N"] * c["E"]
    row_bytes = c["H"] * (4 if c["dt"].startswith("float4") else 8 if "8" in c["dt"] or c["dt"] == "int8"
                          else 16) // 8
    A = int(max(NE, min(3 * NE + int(rng.integers(0, 5000)), (64 << 20) // max(1, row_bytes))))
    scale_cols = {"none": 0, "f32_a": 1, "f32_as": 3, "e8m0": 2 * int(rng.integers(1, 60))}[c["sl"]]
    p = workloads.make_problem(rng, A=A, H=c["H"], N=c["N"], E=c["E"], token_dtype=c["dt"],
                               count_dtype=np.int64 if c["i64"] else np.int32, scale_layout=c["sl"],
                               scale_cols=scale_cols, has_topk=c["topk"], idx_type=c["idx"])
    ref = oracle.run_problem(p)
    # a source at an odd byte offset can only be read on the vector path
    path = m.MRR_PATH_VECTOR if c["off"] else None
    assert_bit_exact(run_gpu_multi(p, layout=c["layout"], path=path, src_offset=c["off"],
                                   sc_offset=(c["case"] * 3) % 8, tk_offset=(c["case"] * 5) % 4,
                                   spare_rows=c["case"] % 7), ref, p)
    if c["off"] == 0:
        assert_bit_exact(run_gpu_multi(p, layout=c["layout"], path=m.MRR_PATH_VECTOR), ref, p)


@pytest.mark.parametrize("edit", [dict(chunk_bytes=4096, stages=2), dict(sched=0), dict(static_chunks=1),
                                  dict(grid=1), dict(block=1024, grid=7), dict(hints=3)])
def test_bulk_pipeline_stress(edit):
    """Small chunks that straddle many rank boundaries, static and dynamic scheduling, one CTA."""
    rng = np.random.default_rng(77)
    p = workloads.make_problem(rng, A=6000, H=256, N=24, E=5, token_dtype="bfloat16", scale_layout="f32_as",
                               scale_cols=2, has_topk=True)
    assert_bit_exact(run_gpu_multi(p, path=m.MRR_PATH_BULK, edit=edit), oracle.run_problem(p), p)


@pytest.mark.parametrize("N,E", [(8, 8), (90, 60)], ids=["fused-scan", "scan-kernel"])
@pytest.mark.parametrize("fault", ["null", "misaligned", "capacity"])
def test_bad_sources_are_refused_then_recovered(N, E, fault):
    """The kernels check every rank's pointers and row count before they read any source: a
    refused call moves nothing and reports MRR_ERR_SOURCE; the next valid call is bit-exact."""
    rng = np.random.default_rng(N + E)
    p = workloads.make_problem(rng, A=3 * N * E + 100, H=512, N=N, E=E, token_dtype="bfloat16",
                               scale_layout="f32_a", scale_cols=1, has_topk=True)
    rows = np.diff(rank_rows(p.counts))
    kw = {"null": dict(null_rank=N // 2),
          "misaligned": dict(src_offset=8, path=m.MRR_PATH_BULK),
          "capacity": dict(rows_override=np.where(np.arange(N) == N - 1, rows - 1, rows))}[fault]
    ws = DevBuf(1 << 20, "cuda:0")
    bad = run_gpu_multi(p, workspace=ws, **kw)
    assert bad["status"] == m.MRR_ERR_SOURCE, m.mrr_status_str(bad["status"])
    assert bad["guards_intact"] and bad["inputs_intact"]
    assert (bad["permute_tokens"] == 0xA5).all()
    assert (bad["permute_token_idx"].view(np.uint8) == 0xA5).all()
    assert_bit_exact(run_gpu_multi(p, workspace=ws), oracle.run_problem(p), p)


def test_counts_are_trusted_without_capacities():
    rng = np.random.default_rng(91)
    p = workloads.make_problem(rng, A=5000, H=64, N=6, E=7, token_dtype="float16", scale_layout="e8m0",
                               scale_cols=6, has_topk=False, idx_type=1)
    assert_bit_exact(run_gpu_multi(p, rows_given=False), oracle.run_problem(p), p)


def test_inverse_plan_is_refused():
    p = workloads.config(1)
    out = run_gpu_multi(p, edit=dict(direction=1), expect_host_status=m.MRR_ERR_PLAN)
    assert out["host_status"] == m.MRR_ERR_PLAN


def test_torch_level_call_matches_single_source():
    import torch

    p = workloads.config(3)
    d = torch.device("cuda:0")
    bounds = rank_rows(p.counts)
    tok = torch.from_numpy(p.tokens.copy()).view(torch.bfloat16).reshape(p.A, p.H).to(d)
    sc = torch.from_numpy(p.scales.copy()).view(torch.float32).reshape(p.A, 4).to(d)
    tw = torch.from_numpy(p.topk.copy()).reshape(p.A, 1).to(d)
    cnt = torch.from_numpy(p.counts).to(d)
    parts = lambda t: [t[bounds[i]:bounds[i + 1]].clone() for i in range(p.N)]
    got = m.moe_re_routing_multi(parts(tok), cnt, per_token_scales=parts(sc), expert_topk_weight=parts(tw),
                                 idx_type=1, check_status=True)
    want = m.moe_re_routing(tok, cnt, per_token_scales=sc, expert_topk_weight=tw, idx_type=1, check_status=True)
    for a, b in zip(got, want):
        assert a.shape == b.shape and a.dtype == b.dtype
        assert torch.equal(a.view(torch.uint8) if a.dtype.is_floating_point else a,
                           b.view(torch.uint8) if b.dtype.is_floating_point else b)
    # counts that do not fit a rank's tensor are refused on the device: rank 2's tensor loses a
    # row and the last rank's gains one, so the rows still sum to A
    moved = parts(tok)
    moved[2] = moved[2][:-1].clone()
    moved[-1] = torch.cat([moved[-1], tok[:1]])
    with pytest.raises(m.MrrError) as err:
        m.moe_re_routing_multi(moved, cnt, check_status=True)
    assert err.value.code == m.MRR_ERR_SOURCE
