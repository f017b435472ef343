"""GPU test of fp8q_gemm_noalloc, the GEMM entry point for callers that cannot
allocate device memory (it keeps its stream-K scratch in an array inside the
library).  Its output must match the workspace GEMM (fp8q_gemm_ws, given a
caller-allocated workspace) within the GEMM tolerance, on two calls in a row.
This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import assert_gemm_close, bf16_ulp, cpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,bmode,out", [
    (512, 512, 8192, 0, torch.bfloat16),   # 8 tiles of 64 K blocks: stream-K cuts every tile
    (384, 256, 5120, 1, torch.float32),    # weight-gradient form (1x128 scales on both sides)
])
def test_noalloc_matches_workspace_gemm(oracle, M, N, K, bmode, out):
    import fp8_fine_grained_21_b300 as fq

    fq.load()
    if bmode == 0:
        A = fi.gaussian((M, K), fi.rng_for(M + K, 0), 1.0, 0.001, 100.0, bf16=False)
        B = fi.gaussian((N, K), fi.rng_for(M + K, 1), 0.02, bf16=False)
        A8, sA = oracle.quant_1x128(A)
        B8, sB = oracle.quant_128x128(B)
    else:
        A = fi.gaussian((K, M), fi.rng_for(M + K, 0), 1.0, 0.001, 100.0, bf16=False)
        B = fi.gaussian((K, N), fi.rng_for(M + K, 1), 1.0, 0.001, 100.0, bf16=False)
        A8, sA = oracle.quant_128x1(A)
        B8, sB = oracle.quant_128x1(B)
    dA8, dsA, dB8, dsB = to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB)
    ws = torch.zeros(fq.fp8q_gemm_workspace_size(), dtype=torch.uint8, device="cuda")
    C_ws = torch.empty((M, N), dtype=out, device="cuda")
    fq.fp8q_gemm_ws(dA8, dsA, dB8, dsB, C_ws, bmode, ws)
    assert fq.fp8q_get_device_status() == 0
    # tolerance: 1e-5 * sum_k |a_k b_k| (plus one BF16 ulp of the value for BF16
    # output) between the two entry points, and both against the oracle
    Cref, Cabs = oracle.gemm(A8, sA, B8, sB, bmode=bmode)
    bf16 = out == torch.bfloat16
    ref = cpu(C_ws).astype(np.float64)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=out, device="cuda")
        fq.fp8q_gemm_noalloc(dA8, dsA, dB8, dsB, C, bmode)
        assert fq.fp8q_get_device_status() == 0
        got = cpu(C).astype(np.float64)
        bound = 1e-5 * Cabs + (bf16_ulp(ref) if bf16 else 0.0)
        bad = np.abs(got - ref) > bound
        assert not bad.any(), "call %d: %d entries differ from fp8q_gemm_ws beyond tolerance" % (
            call, int(bad.sum()))
        assert_gemm_close(got, Cref, Cabs, bf16, "noalloc call %d" % call)
