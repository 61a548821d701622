"""GPU parity of the two API variants: expert_token_num in cumsum mode (expert_token_num_type 0)
and the v1 entry point (mrr_v1_run, the torch_npu.npu_moe_re_routing subset), through the C ABI,
bit for bit against the oracle and against mrr_v2_run."""
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


@pytest.mark.parametrize("shape", [(64, 128, 4, 4, np.int32), (16384, 7168, 16, 16, np.int32),
                                   (3000, 256, 8, 32, np.int64), (9000, 64, 80, 64, np.int64),
                                   (40, 21, 4, 2, np.int32)])
@pytest.mark.parametrize("path", [None, m.MRR_PATH_VECTOR])
def test_cumsum_mode(shape, path):
    A, H, N, E, cdt = shape
    p = workloads.make_problem(np.random.default_rng(A + E), A=A, H=H, N=N, E=E, token_dtype="int8",
                               count_dtype=cdt, scale_layout="f32_a", scale_cols=1)
    p.expert_token_num_type = 0
    ref = oracle.run_problem(p)
    assert int(ref["expert_token_num"][-1]) == A
    assert_bit_exact(run_gpu(p, path=path), ref, p)


def _v1_call(p, with_scales, dev):
    import torch

    code = m.DTYPE_CODES[p.token_dtype]
    tok, cnt = DevBuf.of(p.tokens, dev), DevBuf.of(p.counts, dev)
    sc = DevBuf.of(p.scales, dev) if with_scales else None
    out_tok, out_sc = DevBuf(p.A * p.row_bytes, dev), DevBuf(4 * p.A, dev)
    idx, etn = DevBuf(4 * p.A, dev), DevBuf(p.E * p.counts.dtype.itemsize, dev)
    st, plan = m.mrr_v2_plan(p.A, p.H, code, p.N, p.E, p.count_is_i64,
                             m.MRR_SCALE_F32_A if with_scales else m.MRR_SCALE_NONE, 1, False, 1, 0, 0)
    assert st == m.MRR_OK
    ws = DevBuf(plan.workspace_bytes, dev)
    s = torch.cuda.current_stream().cuda_stream
    st = m.mrr_v1_run(tok.ptr, code, p.A, p.H, cnt.ptr, p.count_is_i64, p.N, p.E,
                      None if sc is None else sc.ptr, out_tok.ptr, out_sc.ptr, idx.ptr, etn.ptr, 1, 0,
                      ws.ptr, ws.n, s)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    assert m.mrr_v2_read_status(ws.ptr, ws.n, s) == m.MRR_OK
    return {"permute_tokens": out_tok.host().reshape(p.A, -1),
            "permute_scales": out_sc.host().reshape(p.A, 4) if with_scales else None,
            "permute_token_idx": idx.host().view(np.int32),
            "expert_token_num": etn.host().view(p.counts.dtype),
            "guards": all(b.guards_intact() for b in (out_tok, out_sc, idx, etn))}


@pytest.mark.parametrize("k,with_scales", [(2, True), (2, False)])
def test_v1_on_the_v1_example_workload(k, with_scales):
    """The v1 page's own usage example shape: int8 A=16384, H=7168, 16 x 16 skewed counts."""
    p = workloads.config(k)
    ref = oracle.run(p.tokens, p.counts, scales=p.scales if with_scales else None, idx_type=0)
    got = _v1_call(p, with_scales, "cuda:0")
    assert got["guards"]
    assert np.array_equal(got["permute_tokens"], ref["permute_tokens"])
    assert np.array_equal(got["permute_token_idx"], ref["permute_token_idx"])
    assert np.array_equal(got["expert_token_num"], ref["expert_token_num"])
    if with_scales:
        assert np.array_equal(got["permute_scales"], ref["permute_scales"])


@pytest.mark.parametrize("dt", ["float16", "bfloat16"])
def test_v1_matches_v2(dt):
    p = workloads.make_problem(np.random.default_rng(77), A=2000, H=1024, N=8, E=8, token_dtype=dt,
                               count_dtype=np.int64, scale_layout="f32_a", scale_cols=1, has_topk=False)
    v2 = run_gpu(p)
    v1 = _v1_call(p, True, "cuda:0")
    for k in ("permute_tokens", "permute_scales", "permute_token_idx", "expert_token_num"):
        assert np.array_equal(v1[k], v2[k]), k


def test_v1_torch_call():
    import torch

    p = workloads.config(1)
    d = torch.device("cuda:0")
    tok = torch.from_numpy(p.tokens.copy()).view(torch.bfloat16).reshape(p.A, p.H).to(d)
    cnt = torch.from_numpy(p.counts).to(d)
    sc = torch.from_numpy(p.scales.copy()).view(torch.float32).reshape(p.A).to(d)
    a = m.moe_re_routing_v1(tok, cnt, per_token_scales=sc, check_status=True)
    b = m.moe_re_routing(tok, cnt, per_token_scales=sc, check_status=True)
    assert len(a) == 4
    for x, y in zip(a, b[:4]):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    with pytest.raises(m.MrrError):
        m.moe_re_routing_v1(tok, cnt, idx_type=1)
