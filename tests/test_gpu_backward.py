"""GPU parity of the backward-pass pieces ("Six Reasons Deepseek Ai Is A Waste
Of Time", para. 3): regrouping the stored 1x128 FP8 activation tiles into 128x1
tiles (bytes and scales bit-exact against the oracle), the FP8 weight transpose
(byte-exact), and the data-gradient GEMM dX = dY W built from them (within the
GEMM tolerance)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import assert_gemm_close, cpu, to_dev
from test_gpu_quant import assert_bytes_equal, assert_scales_equal, special_tile_input
from test_oracle_retile import exact_tiles

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("T,C", [(128, 128), (256, 384), (640, 1024)])
def test_retile_matches_oracle(fq, oracle, bf16, T, C):
    x = special_tile_input(T, C, bf16, seed=T + 7 * C)
    q, s = fq.quant_act_1x128(to_dev(x))
    qT, sT = fq.retile_1x128_to_128x1(q, s)
    qo, so = oracle.quant_1x128(x)
    qTo, sTo = oracle.retile_1x128_to_128x1(qo, so)
    assert_bytes_equal(cpu(qT), qTo, "qT")
    assert_scales_equal(cpu(sT), sTo, "sT")


def test_retile_exact_tiles_equal_direct_128x1(fq, oracle):
    x = exact_tiles(oracle, 384, 256, seed=9)
    q, s = fq.quant_act_1x128(to_dev(x))
    qT, sT = fq.retile_1x128_to_128x1(q, s)
    q2, s2 = fq.quant_act_128x1(to_dev(x))
    assert torch.equal(qT, q2) and torch.equal(sT, s2)


@pytest.mark.slow
def test_retile_wgrad_workload_sampled(fq, oracle):
    """dY[8192][7168]: forward-quantized 1x128, regrouped; three 128-channel
    groups checked against the oracle (a group depends only on its columns)."""
    d = fi.make("wgrad")
    dY = d["dY"]
    q, s = fq.quant_act_1x128(to_dev(dY))
    qT, sT = fq.retile_1x128_to_128x1(q, s)
    qg, sg, qTg, sTg = cpu(q), cpu(s), cpu(qT), cpu(sT)
    for g in (0, 23, 55):
        cols = slice(g * 128, g * 128 + 128)
        qTo, sTo = oracle.retile_1x128_to_128x1(np.ascontiguousarray(qg[:, cols]),
                                                np.ascontiguousarray(sg[g:g + 1]))
        assert_bytes_equal(qTg[cols], qTo, "qT group %d" % g)
        assert_scales_equal(sTg[:, cols], sTo, "sT group %d" % g)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 640), (2048, 7168)])
def test_transpose_w_exact(fq, N, K):
    rng = np.random.default_rng(N + K)
    q = rng.integers(0, 256, (N, K), dtype=np.uint8)
    s = rng.random((N // 128, K // 128), dtype=np.float32)
    qT, sT = fq.transpose_w_128x128(to_dev(q), to_dev(s))
    assert np.array_equal(cpu(qT), q.T)
    assert np.array_equal(cpu(sT), s.T)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_dgrad_gemm(fq, oracle, out):
    """dX[T][K] = dY[T][N] W[N][K]: dY quantized 1x128 along N, W 128x128 and
    transposed; the GEMM's inner dimension is N."""
    T, N, K = 512, 384, 640
    dY = fi.gaussian((T, N), fi.rng_for(31, 0), 1.0, 0.001, 100.0)
    W = fi.gaussian((N, K), fi.rng_for(31, 1), 0.02)
    a8, sa = fq.quant_act_1x128(to_dev(dY))
    w8, sw = fq.quant_w_128x128(to_dev(W))
    wT, swT = fq.transpose_w_128x128(w8, sw)
    dX = fq.gemm(a8, sa, wT, swT, out_dtype=out)
    assert fq.fp8q_get_device_status() == 0
    A8o, sAo = oracle.quant_1x128(dY)
    W8o, sWo = oracle.quant_128x128(W)
    Cref, Cabs = oracle.gemm(A8o, sAo, np.ascontiguousarray(W8o.T), np.ascontiguousarray(sWo.T))
    # the oracle's transposed-operand GEMM agrees with a plain FP64 product of
    # the dequantized operands (an independent route through numpy's matmul)
    Wd = oracle.e4m3_decode(W8o) * np.repeat(np.repeat(sWo.astype(np.float64), 128, 0), 128, 1)
    plain = oracle.dequant_1x128(A8o, sAo) @ Wd
    assert np.allclose(plain, Cref, rtol=1e-12, atol=1e-12 * np.abs(Cref).max())
    assert_gemm_close(cpu(dX), Cref, Cabs, out == torch.bfloat16, "dgrad")
