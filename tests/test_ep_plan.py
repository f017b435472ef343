"""Host side of the expert-parallel MoE data path (FP8 dispatch, BF16
combine; "Six Reasons Deepseek Ai Is A Waste Of Time", para. 4), on CPU:
the per-expert row counts are exchanged between two gloo ranks and each rank
computes its receive layout; the layouts are checked against a brute-force
simulation of every rank's rows, built here from the routing of all ranks.

What the layout must satisfy (for every receiving rank):
  * it receives, from each source rank in rank order, that rank's rows for
    each local expert in expert order, in the source's (token, slot) order;
  * received row i of the pair (source w, local expert e) lands at A8 row
    m_offsets[e] + (rows of e from sources before w) + (its index within w);
  * each expert's rows are contiguous from m_offsets[e], and m_offsets steps
    by the rows rounded up to a multiple of 128."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

W, EL, T, K = 2, 5, 300, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def routing(rank):
    """Rank `rank`'s synthetic top-k routing: Zipf-skewed distinct experts."""
    rng = np.random.default_rng(100 + rank)
    p = np.arange(1, W * EL + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    return np.stack([rng.choice(W * EL, size=K, replace=False, p=p) for _ in range(T)])


def send_rows(ids):
    """Brute force of the send order: (token, slot) pairs sorted by expert,
    then token, then slot."""
    entries = [(int(ids[t, j]), t, j) for t in range(T) for j in range(K)]
    return sorted(entries)


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=W)
    from fp8_fine_grained_21_b300 import ep

    ids = routing(rank)
    counts = np.bincount(ids.reshape(-1), minlength=W * EL)
    by_dest, send_splits = ep.plan_send(counts, W)
    recv_counts = ep.exchange_counts(by_dest, None, torch.device("cpu"))
    plan = ep.plan_recv(recv_counts)
    out[rank] = {"send_splits": send_splits.tolist(), "recv_counts": recv_counts.tolist(),
                 "recv_splits": plan.recv_splits.tolist(), "src_off": plan.src_off.tolist(),
                 "dest_base": plan.dest_base.tolist(), "rows_e": plan.rows_e.tolist(),
                 "m_offsets": plan.m_offsets.tolist(), "Mp": plan.Mp}
    dist.destroy_process_group()


def test_two_rank_receive_layout():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(_free_port(), out), nprocs=W, start_method="spawn",
                       join=True)
    sends = {r: send_rows(routing(r)) for r in range(W)}
    for d in range(W):
        got = out[d]
        # brute force: the rows rank d receives, in receive order, and their expert
        recv = [(w, e, t, j) for w in range(W) for (e, t, j) in sends[w]
                if d * EL <= e < (d + 1) * EL]
        assert got["recv_splits"] == [sum(1 for r in recv if r[0] == w) for w in range(W)]
        assert sum(got["recv_splits"]) == len(recv)
        for w in range(W):       # what rank w sends to d is what d says it receives from w
            assert out[w]["send_splits"][d] == got["recv_splits"][w]
        rows_e = [sum(1 for r in recv if r[1] - d * EL == e) for e in range(EL)]
        assert got["rows_e"] == rows_e
        pad = [(n + 127) // 128 * 128 for n in rows_e]
        assert got["m_offsets"] == list(np.concatenate([[0], np.cumsum(pad)]))
        assert got["Mp"] == sum(pad)
        # destination row of every received row, through the layout tables
        src_off, dest_base = got["src_off"], got["dest_base"]
        dest = []
        for i in range(len(recv)):
            b = max(bb for bb in range(len(dest_base)) if src_off[bb] <= i)
            dest.append(dest_base[b] + i - src_off[b])
        # brute force: expert e's rows, in receive order, fill m_offsets[e] upward
        for e in range(EL):
            mine = [dest[i] for i, r in enumerate(recv) if r[1] - d * EL == e]
            start = got["m_offsets"][e]
            assert mine == list(range(start, start + len(mine)))
        assert len(set(dest)) == len(dest)


def test_single_rank_plan_is_the_identity_exchange():
    from fp8_fine_grained_21_b300 import ep

    ids = routing(0)
    counts = np.bincount((ids % EL).reshape(-1), minlength=EL)   # every expert local
    by_dest, send_splits = ep.plan_send(counts, 1)
    plan = ep.plan_recv(by_dest)
    assert plan.recv_splits.tolist() == send_splits.tolist() == [T * K]
    assert plan.src_off.tolist() == [0] + list(np.cumsum(counts))
    # one source: each expert's first row is its m_offsets entry
    assert plan.dest_base.tolist() == plan.m_offsets[:-1].tolist()
