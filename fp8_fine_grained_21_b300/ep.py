"""Expert-parallel MoE layer with FP8 dispatch and BF16 combine, around the
library's grouped FP8 GEMM ("Six Reasons Deepseek Ai Is A Waste Of Time",
para. 4: activations are quantized to FP8 before they are dispatched to the
experts' up projection; the combine stays in BF16).

Experts are numbered rank-major: rank d of a group of W ranks owns experts
d*E_local .. (d+1)*E_local - 1.  The device work -- 1x128 quantization,
routing, packing, unpacking into the grouped GEMM's layout, the grouped GEMM,
gathering the results back into arrival order and the gate-weighted combine
-- runs in the library's kernels.  This module holds the host side: the
receive layout computed from the exchanged per-expert row counts (a few
integers per source rank and local expert), and the exchanges themselves,
which are torch.distributed all-to-alls of the packed FP8 rows and of the
BF16 results into buffers on this rank's device.  With one rank the
exchanges are the identity.
"""
from dataclasses import dataclass

import numpy as np
import torch

from . import (BSCALE_BLOCK128, fp8q_ep_combine, fp8q_ep_gather, fp8q_ep_pack,
               fp8q_ep_route, fp8q_ep_row_bytes, fp8q_ep_unpack, fp8q_gemm_grouped_ws,
               quant_act_1x128, workspace)


@dataclass
class RecvPlan:
    """Layout of the rows a rank receives: from each source rank w (in rank
    order) the rows it routed to each local expert e (in expert order); block
    b = w * E_local + e.
      recv_splits [W]   rows received from each source
      src_off [nb+1]    start of block b in the receive order
      dest_base [nb]    row of A8 where block b's first row goes
      rows_e [El]       rows of local expert e
      m_offsets [El+1]  start of expert e's rows in A8; each expert's rows
                        padded with zero rows to a multiple of 128
      Mp                rows of A8 (m_offsets[El])"""
    recv_splits: np.ndarray
    src_off: np.ndarray
    dest_base: np.ndarray
    rows_e: np.ndarray
    m_offsets: np.ndarray
    Mp: int


def plan_send(counts, world):
    """Rows this rank sends: counts [E] per expert -> (by_dest [W][E_local],
    send_splits [W]); the send order is expert-major, so destination d's rows
    are contiguous."""
    counts = np.asarray(counts, np.int64)
    if counts.size % world:
        raise ValueError("the number of experts must be a multiple of the number of ranks")
    by_dest = counts.reshape(world, -1)
    return by_dest, by_dest.sum(axis=1)


def plan_recv(recv_counts):
    """recv_counts [W][E_local]: rows source w sends for local expert e ->
    the receive layout (RecvPlan)."""
    rc = np.asarray(recv_counts, np.int64)
    W, El = rc.shape
    rows_e = rc.sum(axis=0)
    padded = (rows_e + 127) // 128 * 128
    m_offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    src_off = np.concatenate([[0], np.cumsum(rc.reshape(-1))]).astype(np.int64)
    before = np.cumsum(rc, axis=0) - rc                 # rows of expert e from earlier sources
    dest_base = (m_offsets[:-1][None, :] + before).reshape(-1).astype(np.int64)
    return RecvPlan(rc.sum(axis=1), src_off, dest_base, rows_e, m_offsets, int(m_offsets[-1]))


def exchange_counts(by_dest, group, device):
    """All-to-all of the per-(destination, local expert) row counts: returns
    recv_counts [W][E_local], row w being what rank w sends here."""
    import torch.distributed as dist

    W, El = by_dest.shape
    send = torch.as_tensor(np.ascontiguousarray(by_dest).reshape(-1), dtype=torch.int64,
                           device=device)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    return recv.cpu().numpy().reshape(W, El)


def _exchange_rows(send, send_splits, recv_splits, group):
    import torch.distributed as dist

    recv = torch.empty((int(np.sum(recv_splits)),) + tuple(send.shape[1:]), dtype=send.dtype,
                       device=send.device)
    dist.all_to_all_single(recv, send, [int(v) for v in recv_splits],
                           [int(v) for v in send_splits], group=group)
    return recv


def dispatch(x, topk_ids, num_experts, stream=None):
    """Quantize the tokens x [T][H] (BF16) per 1x128 tile, route them and pack
    one row per (token, slot).  Returns (send [T*k][row bytes] uint8,
    counts [E] numpy, pos [T][k] int32 on the device)."""
    T, H = x.shape
    k = topk_ids.shape[1]
    q, s = quant_act_1x128(x, stream)
    counts = torch.empty(num_experts, dtype=torch.int32, device=x.device)
    pos = torch.empty((T, k), dtype=torch.int32, device=x.device)
    fp8q_ep_route(topk_ids, num_experts, counts, pos, stream)
    send = torch.empty((T * k, fp8q_ep_row_bytes(H)), dtype=torch.uint8, device=x.device)
    fp8q_ep_pack(q, s, pos, send, stream)
    return send, counts.cpu().numpy().astype(np.int64), pos


def expert_compute(recv, plan, w8, sw, stream=None):
    """Received packed rows -> the grouped GEMM over the local experts (w8
    [E_local][N][H] E4M3, sw [E_local][N/128][H/128]) -> BF16 results in the
    order the rows arrived [R][N]."""
    El, N, H = w8.shape
    dev = w8.device
    R = recv.shape[0]
    out = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    if plan.Mp == 0:
        return out
    t64 = lambda a: torch.as_tensor(a, dtype=torch.int64, device=dev)  # noqa: E731
    src_off, dest_base = t64(plan.src_off), t64(plan.dest_base)
    A8 = torch.empty((plan.Mp, H), dtype=torch.uint8, device=dev)
    sA = torch.empty((H // 128, plan.Mp), dtype=torch.float32, device=dev)
    fp8q_ep_unpack(recv, src_off, dest_base, t64(plan.m_offsets), t64(plan.rows_e), A8, sA, stream)
    Y = torch.empty((plan.Mp, N), dtype=torch.bfloat16, device=dev)
    offs32 = torch.as_tensor(plan.m_offsets, dtype=torch.int32, device=dev)
    fp8q_gemm_grouped_ws(A8, sA, w8, sw, Y, offs32, workspace(dev, stream), stream)
    fp8q_ep_gather(Y, src_off, dest_base, out, stream)
    return out


def combine(back, pos, topk_w, stream=None):
    """back [T*k][N] BF16 (results in the send order) -> out [T][N] BF16 =
    bf16(sum_j topk_w[t][j] * y_tj)."""
    T, k = pos.shape
    out = torch.empty((T, back.shape[1]), dtype=torch.bfloat16, device=back.device)
    fp8q_ep_combine(back, pos, topk_w, out, stream)
    return out


def moe_forward_ep(x, topk_ids, topk_w, w8, sw, group=None, stream=None):
    """One expert-parallel MoE layer on this rank.
      x [T][H] BF16, topk_ids [T][k] int32 (global expert ids, rank-major),
      topk_w [T][k] float32 gate weights,
      w8 [E_local][N][H] uint8 and sw [E_local][N/128][H/128] float32: this
      rank's experts' weights quantized per 128x128 block,
      group: the torch.distributed group of the expert-parallel ranks
      (None: a single rank).
    Returns out [T][N] BF16."""
    import torch.distributed as dist

    world = 1 if group is None else dist.get_world_size(group)
    El = w8.shape[0]
    send, counts, pos = dispatch(x, topk_ids, El * world, stream)
    by_dest, send_splits = plan_send(counts, world)
    if world == 1:
        recv_counts, recv = by_dest, send
    else:
        recv_counts = exchange_counts(by_dest, group, x.device)
        recv = _exchange_rows(send, send_splits, recv_counts.sum(axis=1), group)
    plan = plan_recv(recv_counts)
    results = expert_compute(recv, plan, w8, sw, stream)
    if world == 1:
        back = results
    else:
        back = _exchange_rows(results, plan.recv_splits, send_splits, group)
    return combine(back, pos, topk_w, stream)
