"""Device-side failure detection without faulting the GPU: a bounded wait on
a barrier nothing arrives on runs out, records FP8Q_ERR_TIMEOUT in the sticky
status word, and returns; the status reads once and then clears, and the GPU
and the CUDA context keep working (a GEMM right after is still correct)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import assert_gemm_close, cpu, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(oracle):
    import fp8_fine_grained_21_b300 as fq

    fq.load()
    assert fq.fp8q_get_device_status() in (0, 5)        # start from a clean status word
    assert fq.fp8q_get_device_status() == 0
    fq.fp8q_selftest_wait(1000000)                      # 1 ms limit
    assert fq.fp8q_get_device_status() == 5             # FP8Q_ERR_TIMEOUT
    assert fq.fp8q_get_device_status() == 0             # cleared once read
    # the context is healthy: a GEMM right after is correct
    A = fi.gaussian((256, 512), fi.rng_for(1, 0), bf16=False)
    B = fi.gaussian((256, 512), fi.rng_for(1, 1), bf16=False)
    A8, sA = oracle.quant_1x128(A)
    B8, sB = oracle.quant_128x128(B)
    C = fq.gemm(to_dev(A8), to_dev(sA), to_dev(B8), to_dev(sB), out_dtype=torch.float32)
    assert fq.fp8q_get_device_status() == 0
    Cref, Cabs = oracle.gemm(A8, sA, B8, sB)
    assert_gemm_close(cpu(C), Cref, Cabs, False, "after timeout")


def test_timeout_is_sticky_until_read():
    import fp8_fine_grained_21_b300 as fq

    fq.load()
    fq.fp8q_get_device_status()
    fq.fp8q_selftest_wait(200000)
    fq.fp8q_selftest_wait(200000)                       # a second wait sees the status already set
    torch.cuda.synchronize()
    assert fq.fp8q_get_device_status() == 5
    assert fq.fp8q_get_device_status() == 0
