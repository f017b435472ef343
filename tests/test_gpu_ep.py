"""GPU parity of the expert-parallel MoE data path (FP8 dispatch, BF16
combine; "Six Reasons Deepseek Ai Is A Waste Of Time", para. 4) against the
oracle's moe_ep_reference, on one GPU:
  * fp8q_ep_route: counts and positions exactly those of a stable counting
    sort by expert (the plain definition), including empty experts; an
    out-of-range id is reported and nothing is written;
  * the whole layer on one rank, and with two ranks emulated on this GPU
    (each rank's dispatch, the exchanges done here by slicing and
    concatenating the ranks' buffers in the order the all-to-all would,
    each rank's expert GEMM and combine), against the oracle;
  * pack / unpack round trip: bytes and scales land bit-exact, padding rows
    are zero.
Tolerance of an output element (from the arithmetic): each expert result
y_j is within 1e-5 sum|ab| + 1 BF16 ulp of the exact value (the grouped
GEMM's BF16 bound) and the oracle's bf16(y_j) within half an ulp; the FP32
combine adds at most k * 2^-24 sum_j |w_j y_j|; each side rounds the sum to
BF16 once (half an ulp each):
    |out - ref| <= sum_j |w_j| (1e-5 yabs_j + 2 ulp(y_j))
                   + 1e-6 sum_j |w_j y_j| + ulp(ref) + ulp(sum)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import bf16_ulp, cpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    gates = rng.random((T, k)).astype(np.float32)
    return ids, gates


def experts(oracle, E, N, H, seed):
    W = fi.gaussian((E, N, H), fi.rng_for(seed, 1), 0.02, bf16=False)
    W8 = np.empty((E, N, H), np.uint8)
    sW = np.empty((E, N // 128, H // 128), np.float32)
    for e in range(E):
        W8[e], sW[e] = oracle.quant_128x128(W[e])
    return W8, sW


def assert_moe_close(oracle, out, x, ids, gates, W8, sW, what):
    ref, y, yabs = oracle.moe_ep_reference(x, ids, gates, W8, sW)
    w = np.abs(gates.astype(np.float64))[:, :, None]
    s = np.einsum("tk,tkn->tn", gates.astype(np.float64), y)
    bound = ((w * (1e-5 * yabs + 2 * bf16_ulp(np.abs(y) * 1.01))).sum(axis=1)
             + 1e-6 * (w * np.abs(y)).sum(axis=1) + bf16_ulp(np.abs(ref) * 1.01)
             + bf16_ulp(np.abs(s) * 1.01))
    err = np.abs(cpu(out).astype(np.float64) - ref)
    bad = err > bound
    assert not bad.any(), "%s: %d of %d outputs off, worst %g (bound %g)" % (
        what, int(bad.sum()), bad.size, err[bad].max(), bound[bad][np.argmax(err[bad])])


@pytest.mark.parametrize("T,k,E", [(1000, 3, 17), (64, 1, 4), (0, 2, 8), (513, 8, 256)])
def test_route_is_a_stable_counting_sort(fq, T, k, E):
    ids, _ = routing(T, E, min(k, E), seed=T + E) if T else (np.zeros((0, k), np.int32), None)
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    pos = torch.full((T, ids.shape[1]), -1, dtype=torch.int32, device="cuda")
    fq.fp8q_ep_route(to_dev(ids), E, counts, pos)
    assert fq.fp8q_get_device_status() == 0
    flat = ids.reshape(-1).astype(np.int64)
    want_counts = np.bincount(flat, minlength=E)
    order = np.argsort(flat, kind="stable")            # expert-major, then row-major
    want_pos = np.empty(flat.size, np.int64)
    want_pos[order] = np.arange(flat.size)
    assert np.array_equal(cpu(counts), want_counts)
    assert np.array_equal(cpu(pos).reshape(-1), want_pos)


def test_route_rejects_bad_ids(fq):
    ids = np.array([[0, 1], [2, 9]], np.int32)
    counts = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    pos = torch.full((2, 2), -1, dtype=torch.int32, device="cuda")
    fq.fp8q_ep_route(to_dev(ids), 4, counts, pos)
    assert fq.fp8q_get_device_status() == 7               # FP8Q_ERR_BAD_ROUTING
    assert torch.all(counts == -1).item() and torch.all(pos == -1).item()


def test_pack_unpack_round_trip(fq, oracle):
    from fp8_fine_grained_21_b300 import ep

    T, H, k, E = 200, 384, 2, 3
    x = fi.gaussian((T, H), fi.rng_for(7, 0), 1.0, 0.01, 50.0)
    ids, _ = routing(T, E, k, seed=7)
    send, counts, pos = ep.dispatch(to_dev(x), to_dev(ids), E)
    q, s = oracle.quant_1x128(x)
    by_dest, _ = ep.plan_send(counts, 1)
    plan = ep.plan_recv(by_dest)
    dev = send.device
    t64 = lambda a: torch.as_tensor(a, dtype=torch.int64, device=dev)  # noqa: E731
    A8 = torch.full((plan.Mp, H), 0x5A, dtype=torch.uint8, device=dev)
    sA = torch.full((H // 128, plan.Mp), 3.0, dtype=torch.float32, device=dev)
    fq.fp8q_ep_unpack(send, t64(plan.src_off), t64(plan.dest_base), t64(plan.m_offsets),
                      t64(plan.rows_e), A8, sA)
    assert fq.fp8q_get_device_status() == 0
    A8h, sAh = cpu(A8), cpu(sA)
    posh = cpu(pos)
    for e in range(E):
        ts, js = np.nonzero(ids == e)
        rows = plan.m_offsets[e] + (posh[ts, js] - plan.src_off[e])   # one source: blocks = experts
        assert np.array_equal(A8h[rows], q[ts]) and np.array_equal(sAh[:, rows], s[:, ts])
        pad = np.arange(plan.m_offsets[e] + plan.rows_e[e], plan.m_offsets[e + 1])
        assert np.all(A8h[pad] == 0) and np.all(sAh[:, pad] == 0)


@pytest.mark.parametrize("T,H,N,E,k", [(512, 1024, 768, 8, 2), (300, 512, 256, 5, 3)])
def test_moe_single_rank(fq, oracle, T, H, N, E, k):
    from fp8_fine_grained_21_b300 import ep

    x = fi.gaussian((T, H), fi.rng_for(T + E, 0), 1.0, 0.001, 100.0)
    ids, gates = routing(T, E, k, seed=T + E)
    W8, sW = experts(oracle, E, N, H, seed=T + E)
    out = ep.moe_forward_ep(to_dev(x), to_dev(ids), to_dev(gates), to_dev(W8), to_dev(sW))
    assert fq.fp8q_get_device_status() == 0
    assert_moe_close(oracle, out, x, ids, gates, W8, sW, "one rank")


def test_moe_two_ranks_emulated(fq, oracle):
    """Two ranks on this GPU: each dispatches its own tokens; the all-to-all
    of packed rows and the one of results are done here, as the collective
    would: destination d receives from source 0 then source 1 the rows of
    d's experts (contiguous in each source's send order), and each source
    gets its rows' results back in the order it sent them."""
    from fp8_fine_grained_21_b300 import ep

    Wr, El, H, N, k = 2, 4, 512, 384, 3
    T = [260, 190]
    E = Wr * El
    W8, sW = experts(oracle, E, N, H, seed=31)
    xs = [fi.gaussian((T[r], H), fi.rng_for(31 + r, 0), 1.0, 0.001, 100.0) for r in range(Wr)]
    rt = [routing(T[r], E, k, seed=40 + r) for r in range(Wr)]
    sends, splits, by_dest, poss = [], [], [], []
    for r in range(Wr):
        send, counts, pos = ep.dispatch(to_dev(xs[r]), to_dev(rt[r][0]), E)
        bd, sp = ep.plan_send(counts, Wr)
        sends.append(send); splits.append(sp); by_dest.append(bd); poss.append(pos)
    off = [np.concatenate([[0], np.cumsum(sp)]) for sp in splits]
    results = []
    for d in range(Wr):
        recv_counts = np.stack([by_dest[w][d] for w in range(Wr)])
        recv = torch.cat([sends[w][off[w][d]:off[w][d + 1]] for w in range(Wr)])
        plan = ep.plan_recv(recv_counts)
        res = ep.expert_compute(recv, plan, to_dev(W8[d * El:(d + 1) * El]),
                                to_dev(sW[d * El:(d + 1) * El]))
        results.append((res, np.concatenate([[0], np.cumsum(plan.recv_splits)])))
    for r in range(Wr):
        back = torch.cat([results[d][0][results[d][1][r]:results[d][1][r + 1]] for d in range(Wr)])
        out = ep.combine(back, poss[r], to_dev(rt[r][1]))
        assert fq.fp8q_get_device_status() == 0
        assert_moe_close(oracle, out, xs[r], rt[r][0], rt[r][1], W8, sW, "rank %d" % r)
