"""GPU parity of the push form of the fused receive (mrr_v2_push) against the oracle.

The dispatch ("torch_npu.npu_moe_distribute_dispatch" page: ep_recv_counts) tells each receiver
how many rows every sender sends to each of its local experts; the re-routing ("CANN
ops-transformer MoeReRoutingV2" article, section 计算公式) lays the received rows out
expert-major.  In the push form each sender writes its rows straight to their expert-major place
in every receiver's buffers, at the DstOffset the receiver computed from its count matrix.

The ranks are emulated on one GPU: every receiver's buffers are this GPU's memory, and the
senders' launches run one after another, in a shuffled order (their segments are disjoint).
After all senders, receiver r's outputs must equal, bit for bit, the oracle run on r's rank-major
input (sender 0's rows for r, then sender 1's, ...) with r's count matrix.  Coverage: token
widths with 16-, 8-, 4- and 1-byte rows, scale layouts, top-k, both count types; and the
refusals: a count <= 0, counts that do not sum to S, a receiver whose rows are too few or whose
pointer is NULL (each reported, with no write outside any buffer).
"""
import numpy as np
import pytest

import oracle
import workloads
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def offsets_host(C: np.ndarray):
    """SrcOffset and DstOffset of a receiver's count matrix, from the library's host routine."""
    N, E = C.shape
    c = np.ascontiguousarray(C, np.int64)
    src = np.empty((N, E), np.int64)
    dst = np.empty((N, E), np.int64)
    st = m.mrr_v2_offsets_host(c.ctypes.data, 1, N, E, int(c.sum()), src.ctypes.data, dst.ctypes.data, None)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    return src, dst


class Exchange:
    """N ranks with E local experts each; c[i, r, j] > 0 rows go from sender i to receiver r's
    expert j.  Sender i's rows are a ``workloads.Problem`` with R = N receivers as its ranks, so
    its segment (r, j) sits at the row-major prefix of c[i]."""

    def __init__(self, seed, N, E, rows_max, H, dt, scale_layout="f32_a", scale_cols=1, has_topk=True,
                 count_dtype=np.int32):
        rng = np.random.default_rng(seed)
        self.N, self.E = N, E
        self.c = rng.integers(1, rows_max + 1, size=(N, N, E)).astype(count_dtype)
        self.sends = [workloads.make_problem(rng, A=int(self.c[i].sum()), H=H, N=N, E=E, token_dtype=dt,
                                             counts=np.ascontiguousarray(self.c[i]), scale_layout=scale_layout,
                                             scale_cols=scale_cols, has_topk=has_topk)
                      for i in range(N)]
        p0 = self.sends[0]
        self.rb, self.sb, self.has_topk = p0.row_bytes, p0.scale_row_bytes, has_topk
        self.scales = p0.scales is not None
        self.code, self.sl, self.scale_cols = m.DTYPE_CODES[dt], m.SCALE_CODES[scale_layout], scale_cols
        # receiver r: rank-major input and the oracle's expert-major result
        self.refs, self.A = [], []
        for r in range(N):
            C = np.ascontiguousarray(self.c[:, r, :])
            toks, scs, tks = [], [], []
            for i in range(N):
                p = self.sends[i]
                lo = int(self.c[i, :r].sum())
                hi = lo + int(self.c[i, r].sum())
                toks.append(p.tokens[lo:hi])
                if self.scales:
                    scs.append(p.scales[lo:hi])
                if has_topk:
                    tks.append(p.topk[lo:hi])
            ref = oracle.run(np.concatenate(toks), C, scales=np.concatenate(scs) if self.scales else None,
                             topk=np.concatenate(tks) if has_topk else None, idx_type=0)
            self.refs.append(ref)
            self.A.append(int(C.sum()))


def dev_table(values, device):
    import torch

    return torch.tensor([int(v) for v in values], dtype=torch.int64, device=device)


def run_push(ex: Exchange, *, order=None, rows_override=None, null_receiver=None, counts_edit=None,
             S_delta=0, expect_host=m.MRR_OK):
    """Every sender pushes into guard-banded receiver buffers; returns (statuses, receivers)."""
    import torch

    d = torch.device("cuda:0")
    N, E = ex.N, ex.E
    recv = []
    for r in range(N):
        A = ex.A[r]
        recv.append({"tok": DevBuf(A * ex.rb, d), "sc": DevBuf(A * ex.sb, d) if ex.scales else None,
                     "tk": DevBuf(A * 4, d) if ex.has_topk else None, "idx": DevBuf(A * 4, d)})
    ptrs = lambda key: dev_table([0 if (r == null_receiver and key == "tok") else recv[r][key].ptr
                                  for r in range(N)], d)
    t_tok, t_idx = ptrs("tok"), ptrs("idx")
    t_sc = ptrs("sc") if ex.scales else None
    t_tk = ptrs("tk") if ex.has_topk else None
    rows = dev_table(ex.A if rows_override is None else rows_override, d)
    offs = [offsets_host(np.ascontiguousarray(ex.c[:, r, :])) for r in range(N)]
    statuses = []
    for i in (range(N) if order is None else order):
        p = ex.sends[i]
        counts = p.counts if counts_edit is None else counts_edit(p.counts.copy())
        src_tok = DevBuf.of(p.tokens, d)
        src_sc = DevBuf.of(p.scales, d) if ex.scales else None
        src_tk = DevBuf.of(p.topk, d) if ex.has_topk else None
        cnt = DevBuf.of(np.ascontiguousarray(counts), d)
        dst = DevBuf.of(np.stack([offs[r][1][i] for r in range(N)]), d)
        rsrc = DevBuf.of(np.stack([offs[r][0][i] for r in range(N)]), d)
        ws = DevBuf(4096, d, fill=0x5A)
        s = torch.cuda.current_stream().cuda_stream
        P = lambda b: None if b is None else (b.ptr if isinstance(b, DevBuf) else b.data_ptr())
        st = m.mrr_v2_push(src_tok.ptr, P(src_sc), P(src_tk), ex.code, p.A + S_delta, p.H,
                           cnt.ptr, int(counts.dtype == np.int64), N, E, ex.sl, ex.scale_cols, dst.ptr, rsrc.ptr,
                           t_tok.data_ptr(), P(t_sc), P(t_tk), t_idx.data_ptr(), rows.data_ptr(), ws.ptr, ws.n, s)
        assert st == expect_host, m.mrr_status_str(st)
        if st != m.MRR_OK:
            return statuses, recv
        statuses.append(m.mrr_v2_read_status(ws.ptr, ws.n, s))
        assert src_tok.host().tobytes() == p.tokens.tobytes(), "a send buffer was modified"
    torch.cuda.synchronize()
    return statuses, recv


def assert_received(ex: Exchange, recv):
    for r in range(ex.N):
        ref, b = ex.refs[r], recv[r]
        assert all(x.guards_intact() for x in b.values() if x is not None), f"receiver {r}: guard band written"
        tok = b["tok"].host().reshape(ex.A[r], ex.rb)
        assert np.array_equal(tok, ref["permute_tokens"]), f"receiver {r}: tokens"
        assert np.array_equal(b["idx"].host().view(np.int32), ref["permute_token_idx"]), f"receiver {r}: idx"
        if ex.scales:
            assert np.array_equal(b["sc"].host().reshape(ex.A[r], ex.sb), ref["permute_scales"]), f"{r}: scales"
        if ex.has_topk:
            assert np.array_equal(b["tk"].host().view(np.uint32), ref["permute_topk_weight"].view(np.uint32))


@pytest.mark.parametrize("N,E,rows_max,H,dt,sl,cols,topk,cdt", [
    (2, 1, 5, 128, "bfloat16", "f32_a", 1, True, np.int32),        # 256-byte rows: 16-byte copies
    (4, 3, 20, 7168, "int8", "e8m0", 112, True, np.int64),         # the page's H, e8m0 scales
    (8, 8, 12, 1000, "int8", "f32_as", 3, False, np.int32),        # 1000-byte rows: 8-byte copies
    (3, 5, 9, 250, "float4_e2m1", "none", 0, True, np.int64),      # 125-byte rows: byte copies
    (5, 2, 30, 2, "float16", "f32_a", 1, True, np.int32),          # 4-byte rows
    (16, 16, 4, 512, "float8_e4m3fn", "f32_a", 1, False, np.int32),
])
def test_push_matches_oracle(N, E, rows_max, H, dt, sl, cols, topk, cdt):
    ex = Exchange(N * 100 + E + H, N, E, rows_max, H, dt, sl, cols if sl != "none" else 0, topk, cdt)
    order = list(np.random.default_rng(N + E).permutation(N))
    statuses, recv = run_push(ex, order=order)
    assert all(s == m.MRR_OK for s in statuses), [m.mrr_status_str(s) for s in statuses]
    assert_received(ex, recv)


def test_push_refuses_bad_counts_then_recovers():
    """A count <= 0 (MRR_ERR_COUNT_NONPOS) and counts that do not sum to S (MRR_ERR_COUNT_SUM):
    nothing is written; then the valid exchange runs."""
    ex = Exchange(7, 3, 4, 6, 128, "bfloat16", "f32_a", 1, True)

    def zero(c):
        c[1, 2] = 0
        return c
    statuses, recv = run_push(ex, counts_edit=zero)
    assert statuses and all(s == m.MRR_ERR_COUNT_NONPOS for s in statuses)
    for b in recv:
        assert np.all(b["tok"].host() == 0xA5), "a refused push wrote rows"
    statuses, recv = run_push(ex, S_delta=1)
    assert statuses and all(s == m.MRR_ERR_COUNT_SUM for s in statuses)
    for b in recv:
        assert np.all(b["tok"].host() == 0xA5), "a refused push wrote rows"
    statuses, recv = run_push(ex)
    assert all(s == m.MRR_OK for s in statuses)
    assert_received(ex, recv)


def test_push_refuses_small_or_missing_receiver():
    """A receiver whose buffers hold one row too few, or whose token pointer is NULL: the rows that
    would land past its end (or in it) are not written, the push reports MRR_ERR_DEST, and no
    guard band is touched; the other receivers get their rows."""
    ex = Exchange(11, 4, 3, 8, 256, "float16", "none", 0, False)
    rows = list(ex.A)
    rows[2] -= 1
    statuses, recv = run_push(ex, rows_override=rows)
    assert any(s == m.MRR_ERR_DEST for s in statuses)
    for r in range(ex.N):
        assert all(x.guards_intact() for x in recv[r].values() if x is not None)
        if r != 2:
            assert np.array_equal(recv[r]["tok"].host().reshape(ex.A[r], ex.rb), ex.refs[r]["permute_tokens"])
    statuses, recv = run_push(ex, null_receiver=1)
    assert any(s == m.MRR_ERR_DEST for s in statuses)
    for r in range(ex.N):
        assert all(x.guards_intact() for x in recv[r].values() if x is not None)
        if r != 1:
            assert np.array_equal(recv[r]["tok"].host().reshape(ex.A[r], ex.rb), ex.refs[r]["permute_tokens"])


def test_push_host_refusals():
    """Arguments the host rejects before anything is enqueued."""
    import torch

    d = torch.device("cuda:0")
    ws = DevBuf(4096, d)
    buf = DevBuf(4096, d)
    s = torch.cuda.current_stream().cuda_stream
    bf16 = m.DTYPE_CODES["bfloat16"]
    # R * E above 4096 segments
    assert m.mrr_v2_push(buf.ptr, None, None, bf16, 8192, 8, buf.ptr, 0, 64, 65, m.MRR_SCALE_NONE, 0, buf.ptr,
                         None, buf.ptr, None, None, None, None, ws.ptr, ws.n, s) == m.MRR_ERR_SHAPE
    # missing token destinations
    assert m.mrr_v2_push(buf.ptr, None, None, bf16, 4, 8, buf.ptr, 0, 2, 2, m.MRR_SCALE_NONE, 0, buf.ptr, None,
                         None, None, None, None, None, ws.ptr, ws.n, s) == m.MRR_ERR_NULL
    # an index table without the receivers' source offsets
    assert m.mrr_v2_push(buf.ptr, None, None, bf16, 4, 8, buf.ptr, 0, 2, 2, m.MRR_SCALE_NONE, 0, buf.ptr, None,
                         buf.ptr, None, None, buf.ptr, None, ws.ptr, ws.n, s) == m.MRR_ERR_NULL
    # top-k weights sent with nowhere to go
    assert m.mrr_v2_push(buf.ptr, None, buf.ptr, bf16, 4, 8, buf.ptr, 0, 2, 2, m.MRR_SCALE_NONE, 0, buf.ptr,
                         None, buf.ptr, None, None, None, None, ws.ptr, ws.n, s) == m.MRR_ERR_TOPK_PAIR
    # too small a workspace
    assert m.mrr_v2_push(buf.ptr, None, None, bf16, 4, 8, buf.ptr, 0, 2, 2, m.MRR_SCALE_NONE, 0, buf.ptr, None,
                         buf.ptr, None, None, None, None, ws.ptr, 1024, s) == m.MRR_ERR_WORKSPACE
    # the empty problem: nothing to move, a clean status
    assert m.mrr_v2_push(buf.ptr, None, None, bf16, 0, 8, buf.ptr, 0, 0, 0, m.MRR_SCALE_NONE, 0, buf.ptr, None,
                         buf.ptr, None, None, None, None, ws.ptr, ws.n, s) == m.MRR_OK
    assert m.mrr_v2_read_status(ws.ptr, ws.n, s) == m.MRR_OK
