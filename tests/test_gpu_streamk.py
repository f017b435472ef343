"""GPU tests of the stream-K schedule (GEMM with a workspace): shapes where the
last wave is shared out by K iterations, checked against the CPU oracle within
the GEMM tolerance; repeat calls are bit-identical (pieces are summed in K
order whatever order they finish in); the arrival counters are left zero; the
workspace arguments are checked."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import assert_gemm_close, cpu, to_dev
from test_gpu_gemm import corner_and_random, compact_entries, grouped_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def counters_zero(ws):
    """The counter region: 64 bytes per SM, rounded up to 256 bytes."""
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = (64 * sms + 255) // 256 * 256
    return int(torch.count_nonzero(ws[:n]).item()) == 0


def run_dense(fq, oracle, M, N, K, out, bmode, seed, full=True):
    if bmode == 0:
        A = fi.gaussian((M, K), fi.rng_for(seed, 0), 1.0, 0.001, 100.0, bf16=False)
        B = fi.gaussian((N, K), fi.rng_for(seed, 1), 0.02, bf16=False)
        A8, sA = oracle.quant_1x128(A)
        B8, sB = oracle.quant_128x128(B)
    else:
        A = fi.gaussian((K, M), fi.rng_for(seed, 0), 1.0, 0.001, 100.0, bf16=False)
        B = fi.gaussian((K, N), fi.rng_for(seed, 1), 1.0, 0.001, 100.0, bf16=False)
        A8, sA = oracle.quant_128x1(A)
        B8, sB = oracle.quant_128x1(B)
    dA8, dsA, dB8, dsB = to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB)
    ws = fq.workspace()
    C1 = torch.empty((M, N), dtype=out, device="cuda")
    C2 = torch.empty_like(C1)
    Cdp = torch.empty_like(C1)
    fq.fp8q_gemm_ws(dA8, dsA, dB8, dsB, C1, bmode, ws)
    fq.fp8q_gemm_ws(dA8, dsA, dB8, dsB, C2, bmode, ws)
    fq.fp8q_gemm_ws(dA8, dsA, dB8, dsB, Cdp, bmode, None)
    assert fq.fp8q_get_device_status() == 0
    bf16 = out == torch.bfloat16
    if full:
        Cref, Cabs = oracle.gemm(A8, sA, B8, sB, bmode=bmode)
        assert_gemm_close(cpu(C1), Cref, Cabs, bf16, "stream-K")
        assert_gemm_close(cpu(Cdp), Cref, Cabs, bf16, "whole tiles")
    else:
        rng = np.random.default_rng(seed)
        rows = corner_and_random(M, 16, rng)
        cols = corner_and_random(N, 16, rng)
        mi, ni = compact_entries(rows, cols, rng, extra=1024)
        Cref, Cabs = oracle.gemm_entries(A8, sA, B8, sB, rows[mi], cols[ni], bmode=bmode)
        assert_gemm_close(cpu(C1)[rows[mi], cols[ni]], Cref, Cabs, bf16, "stream-K (sampled)")
        assert_gemm_close(cpu(Cdp)[rows[mi], cols[ni]], Cref, Cabs, bf16, "whole tiles (sampled)")
    assert torch.equal(C1, C2), "stream-K result changed between identical calls"
    assert counters_zero(ws)


@pytest.mark.parametrize("M,N,K,out", [
    (256, 512, 8192, torch.float32),     # 4 tiles of 128x256, 64 K blocks: every tile cut 8 ways
    (384, 256, 5120, torch.bfloat16),    # 3 tiles, 40 K blocks
    (128, 384, 4096, torch.float32),     # 128-wide tiles (N % 256 != 0): 3 tiles, 32 K blocks
    (1024, 1024, 4096, torch.float32),   # 32 tiles: all stream-K
])
def test_streamk_dense(fq, oracle, M, N, K, out):
    run_dense(fq, oracle, M, N, K, out, 0, seed=M + N + K)


def test_streamk_dense_waves_plus_tail(fq, oracle):
    """320 tiles of 64 K blocks on 148 SMs: one whole-tile wave, then the
    other 172 tiles shared out."""
    run_dense(fq, oracle, 5120, 2048, 8192, torch.bfloat16, 0, seed=3, full=False)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_streamk_row_scaled(fq, oracle, out):
    """Weight-gradient form (1x128 scales on both operands), K over tokens."""
    run_dense(fq, oracle, 384, 256, 5120, out, 1, seed=11)


def test_streamk_grouped(fq, oracle):
    sizes = np.array([128, 0, 256, 384, 128])
    N, K = 256, 128 * 48
    offs, A8, sA, B8, sB = grouped_case(oracle, sizes, N, K, seed=21)
    Mtot = A8.shape[0]
    ws = fq.workspace()
    dA8, dsA, dB8, dsB = to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB)
    doffs = to_dev(offs.astype(np.int32))
    C1 = torch.full((Mtot, N), 3.0, dtype=torch.float32, device="cuda")
    C2 = torch.full((Mtot, N), 3.0, dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_grouped_ws(dA8, dsA, dB8, dsB, C1, doffs, ws)
    fq.fp8q_gemm_grouped_ws(dA8, dsA, dB8, dsB, C2, doffs, ws)
    assert fq.fp8q_get_device_status() == 0
    Cref, Cabs = oracle.gemm_grouped(A8, sA, B8, sB, offs)
    assert_gemm_close(cpu(C1), Cref, Cabs, False, "grouped stream-K")
    assert torch.equal(C1, C2)
    assert counters_zero(ws)


def test_workspace_argument_checks(fq):
    n = fq.fp8q_gemm_workspace_size()
    assert n > 64 * torch.cuda.get_device_properties(0).multi_processor_count
    A8 = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    sA = torch.ones((1, 128), device="cuda")
    sB = torch.ones((1, 1), device="cuda")
    C = torch.empty((128, 128), device="cuda")
    small = torch.zeros(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.Fp8qError) as e:
        fq.fp8q_gemm_ws(A8, sA, A8, sB, C, 0, small)
    assert e.value.status == 1                       # FP8Q_ERR_INVALID_ARG
    big = torch.zeros(n + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.Fp8qError) as e:
        fq.fp8q_gemm_ws(A8, sA, A8, sB, C, 0, big[16:16 + n])
    assert e.value.status == 3                       # FP8Q_ERR_MISALIGNED
