"""GPU parity of the quantize kernels against the CPU oracle: E4M3 bytes and
FP32 scales must match bit for bit.  Small cases compare every element;
full-size workloads compare every tile of a seeded random sample (tiles are
independent, so a sampled tile is exact ground truth)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import Guarded, cpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def assert_bytes_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, "%s: %d mismatches, first at %s: gpu %r oracle %r" % (
        what, len(bad), tuple(bad[0]), got[tuple(bad[0])], want[tuple(bad[0])])


def assert_scales_equal(got, want, what):
    assert_bytes_equal(np.asarray(got).view(np.uint32), np.asarray(want).view(np.uint32), what)


def special_tile_input(M, K, bf16, seed):
    """Gaussian data with outliers plus rows that hit the edge cases: an
    all-zero tile, negative zeros, a constant tile, a one-hot tile, tiny
    values (subnormal E4M3 outputs), huge values, exact midpoints."""
    x = fi.gaussian((M, K), fi.rng_for(seed, 0), 1.0, 0.002, 100.0, bf16=False)
    if M >= 8 and K >= 256:
        x[0, :128] = 0.0
        x[1, :128] = -0.0
        x[1, 5] = -0.0
        x[2, 128:256] = -3.0
        x[3, :128] = 0.0
        x[3, 77] = 5.5
        x[4, :128] *= np.float32(1e-30)
        x[5, :128] *= np.float32(1e30)
        x[6, :128] = np.float32(2.0 ** -20)
        x[6, 0] = 7.0                              # inv = 64: exact midpoints below
        x[6, 1:4] = [4.25, 4.75, 3.25]
        x[7, :128] = np.float32(1e-38)             # 448/amax overflows FP32
    return fi.to_bf16_bits(x) if bf16 else x


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("M,K", [(1, 128), (64, 256), (200, 384), (333, 1024)])
def test_quant_1x128_small(fq, oracle, bf16, M, K):
    x = special_tile_input(M, K, bf16, seed=M + K)
    q, s = Guarded((M, K), torch.uint8), Guarded((K // 128, M), torch.float32)
    fq.fp8q_quant_act_1x128(to_dev(x), q.t, s.t)
    q.check("q")
    s.check("s")
    qo, so = oracle.quant_1x128(x)
    assert_bytes_equal(cpu(q.t), qo, "q")
    assert_scales_equal(cpu(s.t), so, "s")


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T,C", [(128, 64), (256, 192), (384, 640)])
def test_quant_128x1_small(fq, oracle, bf16, T, C):
    x = special_tile_input(T, C, False, seed=T * 3 + C)
    x[:128, 0] = 0.0                                # all-zero 128x1 tile
    x[:128, 1] = -2.5                               # constant tile
    x[:128, 2] *= np.float32(1e-35)                 # tiny tile
    x[128:, 3] = 0.0
    x[-1, 3] = -6.0                                 # one-hot in the last token group
    if bf16:
        x = fi.to_bf16_bits(x)
    q, s = Guarded((C, T), torch.uint8), Guarded((T // 128, C), torch.float32)
    fq.fp8q_quant_act_128x1(to_dev(x), q.t, s.t)
    q.check("qT")
    s.check("sT")
    qo, so = oracle.quant_128x1(x)
    assert_bytes_equal(cpu(q.t), qo, "qT")
    assert_scales_equal(cpu(s.t), so, "sT")


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 1024)])
def test_quant_128x128_small(fq, oracle, bf16, N, K):
    x = special_tile_input(N, K, bf16, seed=N * 5 + K)
    q, s = Guarded((N, K), torch.uint8), Guarded((N // 128, K // 128), torch.float32)
    fq.fp8q_quant_w_128x128(to_dev(x), q.t, s.t)
    q.check("q")
    s.check("s")
    qo, so = oracle.quant_128x128(x)
    assert_bytes_equal(cpu(q.t), qo, "q")
    assert_scales_equal(cpu(s.t), so, "s")


def test_quant_tiny_workload_full(fq, oracle):
    d = fi.make("tiny")
    q, s = fq.quant_act_1x128(to_dev(d["A"]))
    qo, so = oracle.quant_1x128(d["A"])
    assert_bytes_equal(cpu(q), qo, "A q")
    assert_scales_equal(cpu(s), so, "A s")
    q, s = fq.quant_w_128x128(to_dev(d["B"]))
    qo, so = oracle.quant_128x128(d["B"])
    assert_bytes_equal(cpu(q), qo, "B q")
    assert_scales_equal(cpu(s), so, "B s")


def _sample_rows(n, k, rng):
    return np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)]))


def check_1x128_rows(fq, oracle, x, rows, what):
    q, s = fq.quant_act_1x128(to_dev(x))
    qg, sg = cpu(q), cpu(s)
    qo, so = oracle.quant_1x128(x[rows])
    assert_bytes_equal(qg[rows], qo, what + " q")
    assert_scales_equal(sg[:, rows], so, what + " s")
    return q, s


def check_128x128_blocks(fq, oracle, w, nblocks, rng, what):
    q, s = fq.quant_w_128x128(to_dev(w))
    qg, sg = cpu(q), cpu(s)
    N, K = w.shape
    for nb in _sample_rows(N // 128, nblocks, rng):
        rows = slice(nb * 128, nb * 128 + 128)
        qo, so = oracle.quant_128x128(w[rows])
        assert_bytes_equal(qg[rows], qo, "%s q block row %d" % (what, nb))
        assert_scales_equal(sg[nb:nb + 1], so, "%s s block row %d" % (what, nb))


def check_128x1_tokens(fq, oracle, x, ntb, rng, what):
    q, s = fq.quant_act_128x1(to_dev(x))
    qg, sg = cpu(q), cpu(s)
    T, C = x.shape
    for tb in _sample_rows(T // 128, ntb, rng):
        toks = slice(tb * 128, tb * 128 + 128)
        qo, so = oracle.quant_128x1(x[toks])
        assert_bytes_equal(qg[:, toks], qo, "%s qT token block %d" % (what, tb))
        assert_scales_equal(sg[tb:tb + 1], so, "%s sT token block %d" % (what, tb))


@pytest.mark.slow
def test_quant_forward_workload(fq, oracle):
    d = fi.make("forward")
    rng = np.random.default_rng(0)
    check_1x128_rows(fq, oracle, d["A"], _sample_rows(d["A"].shape[0], 64, rng), "A")
    check_128x128_blocks(fq, oracle, d["W"], 3, rng, "W")


@pytest.mark.slow
def test_quant_wgrad_workload(fq, oracle):
    d = fi.make("wgrad")
    rng = np.random.default_rng(1)
    check_128x1_tokens(fq, oracle, d["dY"], 3, rng, "dY")
    check_128x1_tokens(fq, oracle, d["X"], 3, rng, "X")


@pytest.mark.slow
def test_quant_accum_workload(fq, oracle):
    d = fi.make("accum")
    rng = np.random.default_rng(2)
    check_1x128_rows(fq, oracle, d["A"], _sample_rows(d["A"].shape[0], 32, rng), "A")
    check_128x128_blocks(fq, oracle, d["B"], 2, rng, "B")


@pytest.mark.slow
def test_quant_grouped_workload(fq, oracle):
    d = fi.make("grouped")
    rng = np.random.default_rng(3)
    check_1x128_rows(fq, oracle, d["A"], _sample_rows(d["A"].shape[0], 64, rng), "A")
    W = d["W"]
    G, N, K = W.shape
    q, s = fq.quant_w_128x128(to_dev(W.reshape(G * N, K)))
    qg, sg = cpu(q), cpu(s)
    for e in (0, 17, G - 1):
        nb = int(rng.integers(0, N // 128))
        rows = slice(e * N + nb * 128, e * N + nb * 128 + 128)
        qo, so = oracle.quant_128x128(W[e, nb * 128:(nb + 1) * 128])
        assert_bytes_equal(qg[rows], qo, "W expert %d" % e)
        assert_scales_equal(sg[e * (N // 128) + nb:e * (N // 128) + nb + 1], so, "sW expert %d" % e)
    torch.cuda.synchronize()


# The quantizers are persistent: a few CTAs per SM walk the tiles in turn
# through a ring of shared-memory stages (3 or 4 deep).  These sizes give
# every CTA more tiles than there are stages, so each stage is refilled and
# its barrier changes phase.  Sampled rows / token blocks / block rows always
# include the last ones, whose tiles are the last each CTA handles.
@pytest.mark.parametrize("bf16", [True, False])
def test_quant_1x128_many_tiles_per_cta(fq, oracle, bf16):
    x = special_tile_input(3840 + 17, 5120, bf16, seed=91)     # 2440 tiles of 64 x 128, ragged
    rng = np.random.default_rng(91)
    check_1x128_rows(fq, oracle, x, _sample_rows(x.shape[0], 48, rng), "A")


@pytest.mark.parametrize("bf16", [True, False])
def test_quant_128x1_many_tiles_per_cta(fq, oracle, bf16):
    x = special_tile_input(5120, 3840, bf16, seed=92)          # 2400 tiles of 128 x 64
    check_128x1_tokens(fq, oracle, x, 3, np.random.default_rng(92), "x")


@pytest.mark.parametrize("bf16", [True, False])
def test_quant_128x128_many_tiles_per_cta(fq, oracle, bf16):
    x = special_tile_input(4096, 5120, bf16, seed=93)          # 1280 blocks of 128 x 128
    check_128x128_blocks(fq, oracle, x, 3, np.random.default_rng(93), "w")
