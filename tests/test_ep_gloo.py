"""The push form of the fused receive on CPU ranks (gloo): the counts exchange and the offsets
each sender needs to write its segments into a receiver's expert-major buffer.

The dispatch ("torch_npu.npu_moe_distribute_dispatch" page: ep_recv_counts, expand_x) hands each
rank the rows its peers send to its local experts; the re-routing ("CANN ops-transformer
MoeReRoutingV2" article, section 计算公式) lays them out expert-major.  In the push form no
receiver re-routes anything: sender i writes its segment for receiver r's expert j at the row
DstOffset_r(i, j) it learned from ``moe_expert_token_gb300.ep.sender_offsets`` (with SrcOffset_r(i, j),
the rank-major rows its segment is at the receiver, for the receiver's gather index).

Each rank here sends seeded payload rows to every rank; the payloads travel with gloo, and the
receiver places every sender's segments at the offsets THAT SENDER computed, never its own.
The assembled buffer and gather index must equal, byte for byte, the oracle's re-routing of the
rank-major concatenation the receiver would otherwise have re-routed, and the per-expert counts the
receiver's own offsets give must equal the oracle's.  No GPU is used: the arithmetic is the
library's host routine and the transport is gloo.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

E_LOCAL = 3          # experts per rank
ROW_BYTES = 24


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _send_plan(rank, world):
    """Seeded counts and payload rows this rank sends: counts[r, j] >= 1 rows to rank r's expert
    j, and for each (r, j) its rows, tagged so that a misplaced row is caught."""
    rng = np.random.default_rng(100 + rank)
    counts = rng.integers(1, 9, size=(world, E_LOCAL)).astype(np.int64)
    rows = {}
    for r in range(world):
        for j in range(E_LOCAL):
            blk = rng.integers(0, 256, size=(int(counts[r, j]), ROW_BYTES), dtype=np.uint8)
            blk[:, 0], blk[:, 1], blk[:, 2] = rank, r, j
            rows[r, j] = blk
    return counts, rows


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import oracle
    from moe_expert_token_gb300 import build, ep

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    build.build()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        counts, rows = _send_plan(rank, world)
        # 1. counts exchange: row i of recv = what rank i sends to this rank's experts
        recv = ep.exchange_counts(torch.from_numpy(counts))
        # 2. every sender learns where its segments land in every receiver's output, and which
        #    rank-major rows they are there
        where_t, src_t = ep.sender_offsets(recv)
        where, src_rows = where_t.numpy(), src_t.numpy()       # [world, E]: row r -> receiver r
        assert np.array_equal(where, ep.sender_dst_offsets(recv).numpy())
        # 3. payloads: to rank r, this rank's rows for r's experts in expert order, with the
        #    offsets it computed for them
        send_rows = [np.concatenate([rows[r, j] for j in range(E_LOCAL)]) for r in range(world)]
        send_counts = [len(x) for x in send_rows]
        got_counts = torch.empty(world, dtype=torch.int64)
        dist.all_to_all_single(got_counts, torch.tensor(send_counts, dtype=torch.int64))
        flat = torch.from_numpy(np.concatenate(send_rows).reshape(-1).copy())
        inbox = torch.empty(int(got_counts.sum()) * ROW_BYTES, dtype=torch.uint8)
        dist.all_to_all_single(inbox, flat, output_split_sizes=[int(c) * ROW_BYTES for c in got_counts],
                               input_split_sizes=[c * ROW_BYTES for c in send_counts])
        off_in = torch.empty(world * E_LOCAL, dtype=torch.int64)
        dist.all_to_all_single(off_in, torch.from_numpy(where.reshape(-1).copy()))
        off_in = off_in.numpy().reshape(world, E_LOCAL)          # row i: sender i's offsets here
        src_in = torch.empty(world * E_LOCAL, dtype=torch.int64)
        dist.all_to_all_single(src_in, torch.from_numpy(src_rows.reshape(-1).copy()))
        src_in = src_in.numpy().reshape(world, E_LOCAL)          # row i: sender i's source rows here
        # 4. the receiver places each sender's segments where the SENDER said
        rc = recv.numpy()
        A = int(rc.sum())
        inbox = inbox.numpy().reshape(A, ROW_BYTES)
        out = np.full((A, ROW_BYTES), 0xEE, np.uint8)
        idx = np.full(A, -1, np.int32)                           # the gather index the senders write
        pos = 0
        for i in range(world):
            for j in range(E_LOCAL):
                n = int(rc[i, j])
                out[off_in[i, j]:off_in[i, j] + n] = inbox[pos:pos + n]
                idx[off_in[i, j]:off_in[i, j] + n] = src_in[i, j] + np.arange(n)
                pos += n
        # 5. against the oracle's re-routing of the rank-major rows this rank received
        ref = oracle.run(inbox, rc)
        _, _, etn = ep.receiver_offsets(recv, A)
        ok = (np.array_equal(out, ref["permute_tokens"])
              and np.array_equal(idx, ref["permute_token_idx"])
              and np.array_equal(etn.numpy(), ref["expert_token_num"].astype(np.int64))
              and np.array_equal(rc, np.stack([_send_plan(i, world)[0][rank] for i in range(world)])))
        q.put((rank, bool(ok), A))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_push_offsets_place_every_segment(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = dict((r, (ok, A)) for r, ok, A in (q.get(timeout=10) for _ in range(world)))
    assert all(ok for ok, _ in got.values()), got


def test_offsets_host_matches_the_oracle_and_refuses_bad_counts():
    import torch

    import oracle
    from moe_expert_token_gb300 import build, ep
    import moe_expert_token_gb300.mrr_v2 as m

    build.build()
    rng = np.random.default_rng(7)
    for N, E in [(1, 1), (2, 3), (5, 4), (16, 16)]:
        for dt in (np.int32, np.int64):
            c = rng.integers(1, 50, size=(N, E)).astype(dt)
            src, dst, etn = ep.receiver_offsets(torch.from_numpy(c), int(c.sum()))
            o_src, o_dst = oracle.offsets(c)
            assert np.array_equal(src.numpy(), o_src) and np.array_equal(dst.numpy(), o_dst)
            assert np.array_equal(etn.numpy(), oracle.expert_token_num(c).astype(np.int64))
    c = np.array([[1, 2], [0, 3]], np.int64)
    with pytest.raises(m.MrrError) as e:
        ep.receiver_offsets(torch.from_numpy(c), 6)
    assert e.value.code == m.MRR_ERR_COUNT_NONPOS
    with pytest.raises(m.MrrError) as e:
        ep.receiver_offsets(torch.from_numpy(np.array([[1, 2], [2, 3]], np.int64)), 9)
    assert e.value.code == m.MRR_ERR_COUNT_SUM
