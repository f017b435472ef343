"""GPU parity of the block-scaled FP8 GEMM (dense, weight-gradient and grouped)
against the CPU oracle, within |C - C_ref| <= 1e-5 sum_k |a_k b_k| (+1 BF16
ulp of C_ref for BF16 output).

Two kinds of case: GEMM-only (the oracle's own quantized bytes and scales are
uploaded, so both sides multiply identical operands) and the whole path
(GPU quantize -> GPU GEMM, against oracle quantize -> oracle GEMM)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import Guarded, assert_gemm_close, cpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def oracle_operands(oracle, A, B, bmode=0):
    A8, sA = oracle.quant_1x128(A)
    if bmode == 0:
        B8, sB = oracle.quant_128x128(B)
    else:
        B8, sB = oracle.quant_1x128(B)
    return A8, sA, B8, sB


def sample_entries(M, N, BN, rng, extra=2048):
    """Every output tile's four corners plus random entries."""
    mi, ni = [], []
    for m0 in range(0, M, 128):
        for n0 in range(0, N, BN):
            for dm, dn in ((0, 0), (127, 0), (0, BN - 1), (127, BN - 1)):
                mi.append(m0 + dm)
                ni.append(min(n0 + dn, N - 1))
    mi = np.concatenate([mi, rng.integers(0, M, extra)])
    ni = np.concatenate([ni, rng.integers(0, N, extra)])
    return mi.astype(np.int64), ni.astype(np.int64)


def run_gemm_only(fq, oracle, A, B, out_dtype, bmode=0, full=True, seed=0, stream_k=True):
    A8, sA, B8, sB = oracle_operands(oracle, A, B, bmode)
    Cgd = Guarded((A8.shape[0], B8.shape[0]), out_dtype, fill=float("nan"))
    fq.fp8q_gemm_ws(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), Cgd.t, bmode,
                    fq.workspace() if stream_k else None)
    assert fq.fp8q_get_device_status() == 0
    Cgd.check("C")
    Cg = cpu(Cgd.t).astype(np.float64)
    bf16 = out_dtype == torch.bfloat16
    if full:
        Cref, Cabs = oracle.gemm(A8, sA, B8, sB, bmode=bmode)
        return assert_gemm_close(Cg, Cref, Cabs, bf16, "gemm")
    M, N = Cg.shape
    mi, ni = sample_entries(M, N, 256 if N % 256 == 0 else 128, np.random.default_rng(seed))
    Cref, Cabs = oracle.gemm_entries(A8, sA, B8, sB, mi, ni, bmode=bmode)
    return assert_gemm_close(Cg[mi, ni], Cref, Cabs, bf16, "gemm (sampled)")


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [
    (128, 128, 128),      # one tile, one K block (first MMA must not accumulate)
    (128, 128, 512),      # tiny workload shape
    (256, 384, 1280),     # 128-wide tiles, odd tile count, 10 K blocks
    (384, 512, 640),      # 256-wide tiles
    (128, 1024, 256),
])
def test_dense_small(fq, oracle, out, M, N, K):
    A = fi.gaussian((M, K), fi.rng_for(M + N, 0), 1.0, 0.001, 100.0, bf16=False)
    B = fi.gaussian((N, K), fi.rng_for(M + N, 1), 0.02, bf16=False)
    run_gemm_only(fq, oracle, A, B, out)
    run_gemm_only(fq, oracle, A, B, out, stream_k=False)


def test_dense_persistent_multi_tile(fq, oracle):
    """More output tiles than SMs: CTAs loop over several tiles and the
    pipeline rings carry across tile boundaries."""
    M, N, K = 4096, 1280, 384          # 32 x 5 = 160 tiles of 128 x 256
    A = fi.gaussian((M, K), fi.rng_for(5, 0), 1.0, 0.001, 100.0, bf16=False)
    B = fi.gaussian((N, K), fi.rng_for(5, 1), 0.02, bf16=False)
    run_gemm_only(fq, oracle, A, B, torch.bfloat16, full=False)
    M, N = 2560, 1152                  # 20 x 9 = 180 tiles of 128 x 128
    A = fi.gaussian((M, K), fi.rng_for(6, 0), bf16=False)
    B = fi.gaussian((N, K), fi.rng_for(6, 1), bf16=False)
    run_gemm_only(fq, oracle, A, B, torch.float32, full=False)


def test_dense_zero_and_constant(fq, oracle):
    M, N, K = 256, 256, 384
    A = np.zeros((M, K), np.float32)
    B = fi.gaussian((N, K), fi.rng_for(7, 1), bf16=False)
    C = fq.gemm(*[to_dev(t) for t in oracle_operands(oracle, A, B)], out_dtype=torch.float32)
    assert torch.count_nonzero(C).item() == 0
    # 7 -> scale 2^-6 and -7/16 -> scale 2^-10 are exact, every byte is +-448, and
    # every partial and sum is exact in FP32: C = K * 7 * (-7/16) exactly
    A = np.full((M, K), 7.0, np.float32)
    Bc = np.full((N, K), -0.4375, np.float32)
    C = fq.gemm(*[to_dev(t) for t in oracle_operands(oracle, A, Bc)], out_dtype=torch.float32)
    assert torch.all(C == K * 7.0 * -0.4375).item()


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("stream_k", [False, True])
def test_wgrad_row_scales_128_wide_tiles(fq, oracle, out, stream_k):
    """Row-scaled B (the weight-gradient form) with N % 256 != 0 takes the
    128-column tile instantiation, whose 1x128 B-scale slots and stream-K
    fix-up slices differ from the 256-column one.  3 x 3 tiles of 40 K
    blocks: with a workspace the stream-K schedule cuts every tile."""
    M, N, K = 384, 384, 5120
    dY = fi.gaussian((K, M), fi.rng_for(31, 0), 1.0, 0.001, 100.0, bf16=False)
    X = fi.gaussian((K, N), fi.rng_for(31, 1), 1.0, 0.001, 100.0, bf16=False)
    A8, sA = oracle.quant_128x1(dY)
    B8, sB = oracle.quant_128x1(X)
    Cgd = Guarded((M, N), out, fill=float("nan"))
    fq.fp8q_gemm_ws(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), Cgd.t, fq.BSCALE_ROW1x128,
                    fq.workspace() if stream_k else None)
    assert fq.fp8q_get_device_status() == 0
    Cgd.check("C")
    Cref, Cabs = oracle.gemm(A8, sA, B8, sB, bmode=1)
    assert_gemm_close(cpu(Cgd.t), Cref, Cabs, out == torch.bfloat16, "wgrad 128-wide tiles")


@pytest.mark.parametrize("stream_k", [True, False])
def test_wgrad_row_scales_scale_slot_reuse(fq, oracle, stream_k):
    """With 128-column tiles the TMA producer can run more than eight K blocks
    ahead of the promotion warps, so it waits on the ring of 1x128 scale
    slots and refills a slot as soon as the last promotion warp releases it.
    The slot is read with ordinary loads and refilled by a bulk copy, so the
    release must order those reads before the copy's write; when it did not,
    the slowest warp read some later B scales of the next block.  Several
    whole 128 x 128 tiles are checked, and every tile's corners."""
    T, M, N = 2048, 2048, 1152
    dY = fi.gaussian((T, M), fi.rng_for(41, 0), 1.0, 0.001, 100.0, bf16=False)
    X = fi.gaussian((T, N), fi.rng_for(41, 1), 1.0, 0.001, 100.0, bf16=False)
    A8, sA = oracle.quant_128x1(dY)
    B8, sB = oracle.quant_128x1(X)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_ws(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), C, fq.BSCALE_ROW1x128,
                    fq.workspace() if stream_k else None)
    assert fq.fp8q_get_device_status() == 0
    Cg = cpu(C).astype(np.float64)
    for tm, tn in ((0, 0), (3, 5), (15, 8), (7, 2), (10, 7)):
        r, c = slice(tm * 128, tm * 128 + 128), slice(tn * 128, tn * 128 + 128)
        Cref, Cabs = oracle.gemm(A8[r], sA[:, r], B8[c], sB[:, c], bmode=1)
        assert_gemm_close(Cg[r, c], Cref, Cabs, False, "tile (%d, %d)" % (tm, tn))
    rows = np.concatenate([np.arange(0, M, 128), np.arange(127, M, 128)])
    cols = np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)])
    mi, ni = np.repeat(rows, len(cols)), np.tile(cols, len(rows))
    Cref, Cabs = oracle.gemm_entries(A8, sA, B8, sB, mi, ni, bmode=1)
    assert_gemm_close(Cg[mi, ni], Cref, Cabs, False, "tile corners")


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_wgrad_row_scales_small(fq, oracle, out):
    T, Nd, Kd = 512, 384, 256
    dY = fi.gaussian((T, Nd), fi.rng_for(8, 0), 1.0, 0.001, 100.0, bf16=False)
    X = fi.gaussian((T, Kd), fi.rng_for(8, 1), 1.0, 0.001, 100.0, bf16=False)
    run_gemm_only(fq, oracle, np.ascontiguousarray(dY.T), np.ascontiguousarray(X.T), out, bmode=1)


def test_wgrad_path_end_to_end(fq, oracle):
    """GPU 128x1 quantize of dY and X, GPU GEMM with 1x128 B scales."""
    T, Nd, Kd = 1024, 512, 256
    dY = fi.gaussian((T, Nd), fi.rng_for(9, 0), 1.0, 0.001, 100.0)
    X = fi.gaussian((T, Kd), fi.rng_for(9, 1), 1.0, 0.001, 100.0)
    a8, sa = fq.quant_act_128x1(to_dev(dY))
    b8, sb = fq.quant_act_128x1(to_dev(X))
    C = fq.gemm(a8, sa, b8, sb, out_dtype=torch.float32, bscale=fq.BSCALE_ROW1x128)
    A8o, sAo = oracle.quant_128x1(dY)
    B8o, sBo = oracle.quant_128x1(X)
    Cref, Cabs = oracle.gemm(A8o, sAo, B8o, sBo, bmode=1)
    assert_gemm_close(cpu(C), Cref, Cabs, False, "wgrad path")


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_forward_path_end_to_end(fq, oracle, out):
    M, N, K = 512, 768, 1024
    A = fi.gaussian((M, K), fi.rng_for(10, 0), 1.0, 0.001, 100.0)
    W = fi.gaussian((N, K), fi.rng_for(10, 1), 0.02)
    a8, sa = fq.quant_act_1x128(to_dev(A))
    w8, sw = fq.quant_w_128x128(to_dev(W))
    C = fq.gemm(a8, sa, w8, sw, out_dtype=out)
    A8o, sAo, B8o, sBo = oracle_operands(oracle, A, W)
    Cref, Cabs = oracle.gemm(A8o, sAo, B8o, sBo)
    assert_gemm_close(cpu(C), Cref, Cabs, out == torch.bfloat16, "forward path")


def grouped_case(oracle, sizes, N, K, seed):
    offs = fi.offsets_from_sizes(sizes)
    Mtot = int(offs[-1])
    G = len(sizes)
    A = fi.gaussian((max(Mtot, 128), K), fi.rng_for(seed, 0), 1.0, 0.001, 100.0, bf16=False)
    W = fi.gaussian((G, N, K), fi.rng_for(seed, 1), 0.02, bf16=False)
    A8, sA = oracle.quant_1x128(A)
    B8 = np.empty((G, N, K), np.uint8)
    sB = np.empty((G, N // 128, K // 128), np.float32)
    for e in range(G):
        B8[e], sB[e] = oracle.quant_128x128(W[e])
    return offs, A8, sA, B8, sB


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sizes,N", [
    ([128, 0, 256, 384], 256),
    ([0, 128, 128, 0, 512, 128, 0, 256], 384),
    ([256], 128),
])
def test_grouped_small(fq, oracle, out, sizes, N):
    K = 384
    offs, A8, sA, B8, sB = grouped_case(oracle, np.array(sizes), N, K, seed=sum(sizes) + N)
    Mtot = A8.shape[0]
    C = torch.full((Mtot, N), 12288.0, dtype=out, device="cuda")
    fq.fp8q_gemm_grouped(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), C,
                         to_dev(offs.astype(np.int32)))
    assert fq.fp8q_get_device_status() == 0
    Cref, Cabs = oracle.gemm_grouped(A8, sA, B8, sB, offs)
    Cg = cpu(C).astype(np.float64)
    rows = np.zeros(Mtot, bool)
    rows[offs[0]:offs[-1]] = True
    assert_gemm_close(Cg[rows], Cref[rows], Cabs[rows], out == torch.bfloat16, "grouped")
    assert np.all(Cg[~rows] == 12288.0)             # rows outside every group untouched


def test_grouped_offsets_not_starting_at_zero(fq, oracle):
    N, K = 256, 256
    offs, A8, sA, B8, sB = grouped_case(oracle, np.array([128, 256, 128, 128]), N, K, seed=77)
    offs2 = offs.copy()
    offs2[0] = 128                                    # group 0 becomes empty, rows 0..127 unowned
    C = torch.full((A8.shape[0], N), -1.0, dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_grouped(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), C,
                         to_dev(offs2.astype(np.int32)))
    assert fq.fp8q_get_device_status() == 0
    Cref, Cabs = oracle.gemm_grouped(A8, sA, B8, sB, offs2)
    Cg = cpu(C).astype(np.float64)
    assert np.all(Cg[:128] == -1.0)
    assert_gemm_close(Cg[128:], Cref[128:], Cabs[128:], False, "grouped offset")


@pytest.mark.parametrize("bad", [[0, 100, 256], [0, 256, 128], [0, 128, 1024]])
def test_grouped_bad_offsets_reported(fq, oracle, bad):
    N, K = 128, 128
    offs, A8, sA, B8, sB = grouped_case(oracle, np.array([128, 128]), N, K, seed=3)
    C = torch.full((A8.shape[0], N), 7.0, dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_grouped(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), C,
                         to_dev(np.array(bad, np.int32)))
    assert fq.fp8q_get_device_status() == 6          # FP8Q_ERR_BAD_GROUPS
    assert fq.fp8q_get_device_status() == 0          # cleared after reading
    assert torch.all(C == 7.0).item()                # nothing written


# ------------------------------------------------------------ full workloads
# The oracle quantizes only what the sampled outputs depend on: 1x128 tiles
# and 128x1 tiles belong to one row (channel), so a row subset is exact; a
# 128x128 block needs its whole 128 rows of W.  Every 128 x 128 output tile
# contributes its four corners; random entries come on top.
def corner_and_random(n, k, rng):
    corners = np.concatenate([np.arange(0, n, 128), np.arange(127, n, 128)])
    return np.unique(np.concatenate([corners, rng.integers(0, n, k)])).astype(np.int64)


def compact_entries(rows, cols, rng, extra=4096):
    """All (row, col) pairs where both are tile corners, plus random pairs,
    as indices into the compact row / column lists."""
    rc = np.flatnonzero((rows % 128 == 0) | (rows % 128 == 127))
    cc = np.flatnonzero((cols % 128 == 0) | (cols % 128 == 127))
    mi = np.repeat(rc, len(cc))
    ni = np.tile(cc, len(rc))
    mi = np.concatenate([mi, rng.integers(0, len(rows), extra)])
    ni = np.concatenate([ni, rng.integers(0, len(cols), extra)])
    return mi.astype(np.int64), ni.astype(np.int64)


def check_sampled(Cg, rows, cols, A8c, sAc, B8c, sBc, bmode, bf16, what, rng):
    """Cg: the GPU result on the host.  A8c/sAc: operand A restricted to `rows`;
    B8c/sBc: operand B restricted to `cols` (compact index spaces)."""
    mi, ni = compact_entries(rows, cols, rng)
    Cref, Cabs = oracle_mod().gemm_entries(A8c, sAc, B8c, sBc, mi, ni, bmode=bmode)
    got = Cg[rows[mi], cols[ni]]
    assert_gemm_close(got, Cref, Cabs, bf16, what)


def oracle_mod():
    import oracle
    return oracle


@pytest.mark.slow
def test_forward_workload_sampled(fq, oracle):
    d = fi.make("forward")
    a8, sa = fq.quant_act_1x128(to_dev(d["A"]))
    w8, sw = fq.quant_w_128x128(to_dev(d["W"]))
    C = fq.gemm(a8, sa, w8, sw, out_dtype=torch.bfloat16)
    assert fq.fp8q_get_device_status() == 0
    rng = np.random.default_rng(11)
    rows = corner_and_random(4096, 32, rng)
    cols = corner_and_random(2048, 32, rng)
    A8o, sAo = oracle.quant_1x128(d["A"][rows])
    B8o, sBo = oracle.quant_128x128(d["W"])
    # columns of the compact B: 1x128-style per-column scales expanded from the blocks
    B8c = np.ascontiguousarray(B8o[cols])
    sBc = np.ascontiguousarray(sBo[cols // 128].T)           # [Kb][n_cols]
    check_sampled(cpu(C), rows, cols, A8o, sAo, B8c, sBc, 1, True, "forward workload", rng)


@pytest.mark.slow
@pytest.mark.parametrize("variant", ["", "positive"])
def test_accum_workload_sampled(fq, oracle, variant):
    d = fi.make("accum", variant=variant)
    a8, sa = fq.quant_act_1x128(to_dev(d["A"]))
    b8, sb = fq.quant_w_128x128(to_dev(d["B"]))
    C = fq.gemm(a8, sa, b8, sb, out_dtype=torch.float32)
    assert fq.fp8q_get_device_status() == 0
    rng = np.random.default_rng(12)
    rows = corner_and_random(1024, 32, rng)
    cols = corner_and_random(1024, 32, rng)
    A8o, sAo = oracle.quant_1x128(d["A"][rows])
    B8o, sBo = oracle.quant_128x128(d["B"])
    B8c = np.ascontiguousarray(B8o[cols])
    sBc = np.ascontiguousarray(sBo[cols // 128].T)
    check_sampled(cpu(C), rows, cols, A8o, sAo, B8c, sBc, 1, False, "accum workload " + variant, rng)


@pytest.mark.slow
def test_wgrad_workload_sampled(fq, oracle):
    d = fi.make("wgrad")
    a8, sa = fq.quant_act_128x1(to_dev(d["dY"]))
    b8, sb = fq.quant_act_128x1(to_dev(d["X"]))
    C = fq.gemm(a8, sa, b8, sb, out_dtype=torch.float32, bscale=fq.BSCALE_ROW1x128)
    assert fq.fp8q_get_device_status() == 0
    rng = np.random.default_rng(13)
    rows = corner_and_random(7168, 32, rng)                  # channels of dY
    cols = corner_and_random(2048, 32, rng)                  # channels of X
    A8o, sAo = oracle.quant_128x1(np.ascontiguousarray(d["dY"][:, rows]))
    B8o, sBo = oracle.quant_128x1(np.ascontiguousarray(d["X"][:, cols]))
    check_sampled(cpu(C), rows, cols, A8o, sAo, B8o, sBo, 1, False, "wgrad workload", rng)


@pytest.mark.slow
def test_grouped_workload_sampled(fq, oracle):
    d = fi.make("grouped")
    A, W, offs = d["A"], d["W"], d["m_offsets"]
    G, N, K = W.shape
    a8, sa = fq.quant_act_1x128(to_dev(A))
    w8, sw = fq.quant_w_128x128(to_dev(W.reshape(G * N, K)))
    C = torch.empty((A.shape[0], N), dtype=torch.bfloat16, device="cuda")
    fq.fp8q_gemm_grouped(a8, sa, w8.view(G, N, K), sw.view(G, N // 128, K // 128), C,
                         to_dev(offs.astype(np.int32)))
    assert fq.fp8q_get_device_status() == 0
    rng = np.random.default_rng(14)
    Cg = cpu(C)
    experts = sorted(set([0, G - 1] + [int(e) for e in rng.integers(0, G, 4)]))
    checked = 0
    for e in experts:
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        # first and last row of every 128-row tile of the group, plus random rows
        rows = np.unique(np.concatenate([np.arange(r0, r1, 128), np.arange(r0 + 127, r1, 128),
                                         rng.integers(r0, r1, 8)])).astype(np.int64)
        nbs = sorted(set([0, N // 128 - 1, int(rng.integers(0, N // 128))]))
        cols = np.concatenate([np.arange(nb * 128, nb * 128 + 128) for nb in nbs]).astype(np.int64)
        A8o, sAo = oracle.quant_1x128(A[rows])
        B8o = np.concatenate([oracle.quant_128x128(W[e, nb * 128:nb * 128 + 128])[0] for nb in nbs])
        sBo = np.concatenate([oracle.quant_128x128(W[e, nb * 128:nb * 128 + 128])[1] for nb in nbs])
        check_sampled(Cg, rows, cols, A8o, sAo, B8o, sBo, 0, True, "grouped expert %d" % e, rng)
        checked += 1
    assert checked >= 2
