"""GPU-side test harness: uploads a ``workloads.Problem`` into guard-banded device buffers,
runs the op through the C ABI (``mrr_v2_run`` or ``mrr_v2_run_plan``) and returns the outputs
as numpy arrays.  Every output buffer sits between two 4 KiB guard bands filled with 0xA5 that
must survive the call (an out-of-bounds write check)."""
from __future__ import annotations

from typing import Optional

import numpy as np

import moe_expert_token_gb300.mrr_v2 as m

GUARD = 4096
FILL = 0xA5


class DevBuf:
    """A device byte buffer of ``n`` bytes at ``GUARD + offset`` inside a guard-banded block."""

    def __init__(self, n: int, device, offset: int = 0, fill: int = FILL):
        import torch

        self.n = int(n)
        self.off = GUARD + offset
        self.t = torch.full((self.n + 2 * GUARD + offset,), fill, dtype=torch.uint8, device=device)

    @classmethod
    def of(cls, arr: Optional[np.ndarray], device, offset: int = 0) -> Optional["DevBuf"]:
        import torch

        if arr is None:
            return None
        raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        b = cls(raw.size, device, offset)
        if raw.size:
            b.t[b.off:b.off + b.n].copy_(torch.from_numpy(raw).to(device))
        return b

    @property
    def ptr(self) -> int:
        return self.t.data_ptr() + self.off

    def host(self) -> np.ndarray:
        return self.t[self.off:self.off + self.n].cpu().numpy()

    def guards_intact(self) -> bool:
        import torch

        lo = self.t[:self.off]
        hi = self.t[self.off + self.n:]
        return bool(torch.all(lo == FILL).item()) and bool(torch.all(hi == FILL).item())


def ptr(b: Optional[DevBuf]):
    return None if b is None else b.ptr


def run_gpu(p, *, path: Optional[int] = None, edit: Optional[dict] = None,
            offsets: Optional[dict] = None, device="cuda:0", counts: Optional[np.ndarray] = None,
            workspace: Optional[DevBuf] = None, expect_host_status: int = m.MRR_OK,
            read_status: bool = True) -> dict:
    """Run problem ``p`` on the GPU through the C ABI.

    path / edit: when given, the launch plan from mrr_v2_plan is edited (path, grid, block,
    chunk_bytes, stages) and the call goes through mrr_v2_run_plan; otherwise mrr_v2_run.
    offsets: byte offsets added to the named buffers (to test unaligned pointers).
    """
    import torch

    offsets = offsets or {}
    c = p.counts if counts is None else counts
    code = m.DTYPE_CODES[p.token_dtype]
    sl = m.SCALE_CODES[p.scale_layout]
    A, H, (N, E) = p.A, p.H, c.shape
    d = torch.device(device)
    tok = DevBuf.of(p.tokens, d, offsets.get("tokens", 0))
    cnt = DevBuf.of(c, d, offsets.get("counts", 0))
    sc = DevBuf.of(p.scales, d, offsets.get("scales", 0))
    tw = DevBuf.of(p.topk, d, offsets.get("topk", 0))
    out_tok = DevBuf(A * p.row_bytes, d, offsets.get("permute_tokens", 0))
    out_sc = None if p.scales is None else DevBuf(A * p.scale_row_bytes, d, offsets.get("permute_scales", 0))
    idx = DevBuf(4 * A, d, offsets.get("idx", 0))
    etn = DevBuf(E * c.dtype.itemsize, d, offsets.get("etn", 0))
    out_tw = None if p.topk is None else DevBuf(4 * A, d, offsets.get("permute_topk", 0))

    st, plan = m.mrr_v2_plan(A, H, code, N, E, c.dtype == np.int64, sl, p.scale_cols,
                             p.topk is not None, p.expert_token_num_type, p.idx_type, d.index or 0)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    if workspace is None:
        workspace = DevBuf(plan.workspace_bytes, d, 0, fill=0x5A)
    # device copies of the inputs, compared on the device after the call (any size)
    in_bufs = [b for b in (tok, cnt, sc, tw) if b is not None]
    in_copies = [b.t[b.off:b.off + b.n].clone() for b in in_bufs]
    stream = torch.cuda.current_stream(d).cuda_stream
    if path is None and not edit:
        st = m.mrr_v2_run(ptr(tok), code, A, H, ptr(cnt), c.dtype == np.int64, N, E, ptr(sc), sl,
                          p.scale_cols, ptr(tw), ptr(out_tok), ptr(out_sc), ptr(idx), ptr(etn),
                          ptr(out_tw), p.expert_token_num_type, p.idx_type, workspace.ptr,
                          workspace.n, stream)
    else:
        if path is not None:
            plan.path = path
        for k, v in (edit or {}).items():
            setattr(plan, k, v)
        st = m.mrr_v2_run_plan(plan, ptr(tok), code, ptr(cnt), ptr(sc), ptr(tw), ptr(out_tok),
                               ptr(out_sc), ptr(idx), ptr(etn), ptr(out_tw),
                               p.expert_token_num_type, workspace.ptr, workspace.n, stream)
    assert st == expect_host_status, m.mrr_status_str(st)
    out = {"host_status": st, "plan": plan.as_dict()}
    if st != m.MRR_OK:
        return out
    if read_status:
        out["status"] = m.mrr_v2_read_status(workspace.ptr, workspace.n, stream)
    torch.cuda.synchronize(d)
    out["permute_tokens"] = out_tok.host().reshape(A, p.row_bytes)
    out["permute_scales"] = None if out_sc is None else out_sc.host().reshape(A, p.scale_row_bytes)
    out["permute_token_idx"] = idx.host().view(np.int32)
    out["expert_token_num"] = etn.host().view(c.dtype)
    out["permute_topk_weight"] = None if out_tw is None else out_tw.host().view(np.float32)
    bufs = [out_tok, out_sc, idx, etn, out_tw]
    out["guards_intact"] = all(b.guards_intact() for b in bufs if b is not None)
    out["inputs_intact"] = all(torch.equal(b.t[b.off:b.off + b.n], c) for b, c in zip(in_bufs, in_copies))
    return out


def assert_bit_exact(gpu: dict, ref: dict, p) -> None:
    """Every output equal byte for byte (tolerance 0: nothing is computed on the payloads)."""
    assert gpu["status"] == m.MRR_OK, m.mrr_status_str(gpu["status"])
    assert gpu["guards_intact"], "an output guard band was overwritten"
    assert gpu["inputs_intact"], "an input buffer was modified"
    assert np.array_equal(gpu["permute_token_idx"], ref["permute_token_idx"]), "permute_token_idx"
    assert np.array_equal(gpu["expert_token_num"], ref["expert_token_num"]), "expert_token_num"
    assert gpu["expert_token_num"].dtype == ref["expert_token_num"].dtype
    if not np.array_equal(gpu["permute_tokens"], ref["permute_tokens"]):
        bad = np.nonzero((gpu["permute_tokens"] != ref["permute_tokens"]).any(axis=1))[0]
        raise AssertionError(f"permute_tokens differ in {bad.size} rows, first {bad[:8].tolist()}")
    if p.scales is not None:
        assert np.array_equal(gpu["permute_scales"], ref["permute_scales"]), "permute_scales"
    if p.topk is not None:
        assert np.array_equal(gpu["permute_topk_weight"].view(np.uint32),
                              ref["permute_topk_weight"].view(np.uint32)), "permute_topk_weight"


def run_gpu_unroute(p, *, path: Optional[int] = None, edit: Optional[dict] = None,
                    offsets: Optional[dict] = None, device="cuda:0",
                    counts: Optional[np.ndarray] = None, workspace: Optional[DevBuf] = None,
                    expect_host_status: int = m.MRR_OK) -> dict:
    """Run the inverse move on the GPU through the C ABI.  The problem's tokens / scales / top-k
    payloads serve as the EXPERT-MAJOR inputs; returns the rank-major outputs."""
    import torch

    offsets = offsets or {}
    c = p.counts if counts is None else counts
    code = m.DTYPE_CODES[p.token_dtype]
    sl = m.SCALE_CODES[p.scale_layout]
    A, H, (N, E) = p.A, p.H, c.shape
    d = torch.device(device)
    pt = DevBuf.of(p.tokens, d, offsets.get("permute_tokens", 0))
    cnt = DevBuf.of(c, d, offsets.get("counts", 0))
    ps = DevBuf.of(p.scales, d, offsets.get("permute_scales", 0))
    pw = DevBuf.of(p.topk, d, offsets.get("permute_topk", 0))
    out_tok = DevBuf(A * p.row_bytes, d, offsets.get("tokens", 0))
    out_sc = None if p.scales is None else DevBuf(A * p.scale_row_bytes, d, offsets.get("scales", 0))
    out_tw = None if p.topk is None else DevBuf(4 * A, d, offsets.get("topk", 0))
    st, plan = m.mrr_v2_unroute_plan(A, H, code, N, E, c.dtype == np.int64, sl, p.scale_cols,
                                     p.topk is not None, d.index or 0)
    assert st == m.MRR_OK, m.mrr_status_str(st)
    assert plan.direction == 1
    if workspace is None:
        workspace = DevBuf(plan.workspace_bytes, d, 0, fill=0x5A)
    stream = torch.cuda.current_stream(d).cuda_stream
    if path is None and not edit:
        st = m.mrr_v2_unroute(ptr(pt), code, A, H, ptr(cnt), c.dtype == np.int64, N, E, ptr(ps), sl,
                              p.scale_cols, ptr(pw), ptr(out_tok), ptr(out_sc), ptr(out_tw),
                              workspace.ptr, workspace.n, stream)
    else:
        if path is not None:
            plan.path = path
        for k, v in (edit or {}).items():
            setattr(plan, k, v)
        st = m.mrr_v2_run_plan(plan, ptr(pt), code, ptr(cnt), ptr(ps), ptr(pw), ptr(out_tok),
                               ptr(out_sc), None, None, ptr(out_tw), 1, workspace.ptr, workspace.n,
                               stream)
    assert st == expect_host_status, m.mrr_status_str(st)
    out = {"host_status": st, "plan": plan.as_dict()}
    if st != m.MRR_OK:
        return out
    out["status"] = m.mrr_v2_read_status(workspace.ptr, workspace.n, stream)
    torch.cuda.synchronize(d)
    out["tokens"] = out_tok.host().reshape(A, p.row_bytes)
    out["scales"] = None if out_sc is None else out_sc.host().reshape(A, p.scale_row_bytes)
    out["topk_weight"] = None if out_tw is None else out_tw.host().view(np.float32)
    out["guards_intact"] = all(b.guards_intact() for b in (out_tok, out_sc, out_tw) if b is not None)
    return out


def assert_unroute_bit_exact(gpu: dict, ref: dict, p) -> None:
    assert gpu["status"] == m.MRR_OK, m.mrr_status_str(gpu["status"])
    assert gpu["guards_intact"], "an output guard band was overwritten"
    if not np.array_equal(gpu["tokens"], ref["tokens"]):
        bad = np.nonzero((gpu["tokens"] != ref["tokens"]).any(axis=1))[0]
        raise AssertionError(f"tokens differ in {bad.size} rows, first {bad[:8].tolist()}")
    if p.scales is not None:
        assert np.array_equal(gpu["scales"], ref["scales"]), "scales"
    if p.topk is not None:
        assert np.array_equal(gpu["topk_weight"].view(np.uint32), ref["topk_weight"].view(np.uint32)), "topk"
