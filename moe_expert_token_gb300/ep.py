"""Host-side exchange steps of the expert-parallel dispatch fused with the re-routing.

The op runs right after the dispatch AlltoAll ("CANN ops-transformer MoeReRoutingV2" article,
section 数据流定位; "torch_npu.npu_moe_distribute_dispatch" page: ep_recv_counts, expand_x).
Two fused forms avoid writing the received rows rank-major and reading them again:

* pull (one GPU reads its peers' rows where they landed): ``mrr_v2_run_multi`` takes one source
  buffer per rank, for instance the per-peer slots of a receive buffer;
* push (every sender writes its rows straight into the receiver's expert-major buffer): sender i
  must know, for each receiver r and each of r's local experts j, the row DstOffset_r(i, j) of
  r's output at which its segment (i, j) starts.

This module holds the two exchanges the push form needs before any row moves, written on
``torch.distributed`` (NCCL between GPUs, gloo on CPU):

1. ``exchange_counts``: every rank sends send_counts[r, j] (rows it sends to rank r's local
   expert j) and receives recv_counts[i, j] (rows rank i sends to its own expert j) -- the count
   matrix of its re-routing, the dispatch page's ep_recv_counts;
2. ``sender_offsets``: every rank computes SrcOffset and DstOffset of its count matrix with the
   library's ``mrr_v2_offsets_host`` (the same prefixes the kernels scan) and returns row i of
   each to rank i, so each rank learns where each of its segments lands in every receiver's
   output (DstOffset) and which rank-major rows they are there (SrcOffset, for the receiver's
   gather index).

After these, sender i moves its rows for receiver r's expert j to rows
[DstOffset_r(i, j), DstOffset_r(i, j) + counts) of r's output: ``mrr_v2_push`` does it with plain
stores into the receivers' buffers (over NVLink, a peer's memory), or an NCCL put can.  The
receiver's per-expert counts come from its own count matrix.  The arithmetic runs in the C
library; this module only moves tensors.
"""
from __future__ import annotations

from . import mrr_v2 as _m


def exchange_counts(send_counts, group=None):
    """send_counts [W, E] int64 (row r: rows this rank sends to rank r's local experts) ->
    recv_counts [W, E] int64 (row i: rows rank i sends to this rank's experts), on the same
    device.  One all_to_all of E values per pair of ranks."""
    import torch
    import torch.distributed as dist

    W = dist.get_world_size(group)
    if send_counts.dim() != 2 or send_counts.shape[0] != W or send_counts.dtype != torch.int64:
        raise ValueError("send_counts must be int64 [world_size, E]")
    src = send_counts.contiguous()
    recv = torch.empty_like(src)
    dist.all_to_all_single(recv.view(-1), src.view(-1), group=group)
    return recv


def receiver_offsets(recv_counts, A: int):
    """SrcOffset, DstOffset ([W, E] int64) and expert_token_num ([E] int64) of this rank's count
    matrix, from the library's host routine (on CPU copies of the tensors)."""
    import torch

    c = recv_counts.detach().to("cpu", torch.int64).contiguous()
    N, E = c.shape
    src = torch.empty(N, E, dtype=torch.int64)
    dst = torch.empty(N, E, dtype=torch.int64)
    etn = torch.empty(E, dtype=torch.int64)
    st = _m.mrr_v2_offsets_host(c.data_ptr(), 1, N, E, int(A), src.data_ptr(), dst.data_ptr(), etn.data_ptr())
    if st != _m.MRR_OK:
        raise _m.MrrError(st, "mrr_v2_offsets_host")
    return src, dst, etn


def sender_offsets(recv_counts, group=None):
    """For the push form: returns (dst, src), each [W, E] int64 on recv_counts' device.  Row r of
    dst holds the rows of rank r's expert-major output at which this rank's segments for r's
    experts 0..E-1 start; row r of src the rows of r's rank-major order they are (what r's gather
    index names).  Every rank computes both for its own count matrix and sends row i to rank i:
    the dst_offsets and recv_src_offsets of ``mrr_v2_push``."""
    import torch
    import torch.distributed as dist

    A = int(recv_counts.sum().item())
    src, dst, _ = receiver_offsets(recv_counts, A)
    both = torch.stack([dst, src], dim=1).to(recv_counts.device).contiguous()   # [W, 2, E]
    back = torch.empty_like(both)
    dist.all_to_all_single(back.view(-1), both.view(-1), group=group)
    return back[:, 0].contiguous(), back[:, 1].contiguous()


def sender_dst_offsets(recv_counts, group=None):
    """The dst half of ``sender_offsets``."""
    return sender_offsets(recv_counts, group)[0]


__all__ = ["exchange_counts", "receiver_offsets", "sender_offsets", "sender_dst_offsets"]
