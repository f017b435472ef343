"""Accumulation precision of the GPU path on the accumulation-stress workload
(A[1024][16384] x B[1024][16384] BF16, all-positive U(0,1) variant, 1x128 /
128x128 quantization, FP32 output), next to the limited-accumulation
emulator.

"Six Reasons Deepseek Ai Is A Waste Of Time", paragraph 2, reports a maximum
relative error of nearly 2% at K = 4096 when tensor-core partials are kept in
a limited-width accumulator; paragraph 3 and the "increased accumulation
precision" section say that promoting the partials to FP32 on the CUDA cores
every 128 elements removes that error.  On all-positive data every product
is non-negative, so sum_k |a_k b_k| = C and the GEMM tolerance
|C - C_ref| <= 1e-5 sum_k |a_k b_k| is a relative bound of 1e-5.  This test
measures, on the same sampled outputs, the GPU path's maximum relative error
at the K = 4096 prefix and at the full K = 16384, and the emulator's without
promotion, and prints the figures (run pytest with -s to see them)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import cpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.slow
def test_accum_positive_error_vs_emulator(oracle):
    import fp8_fine_grained_21_b300 as fq

    fq.load()
    d = fi.make("accum", variant="positive")
    A, B = d["A"], d["B"]
    M, K = A.shape
    N = B.shape[0]
    a8, sa = fq.quant_act_1x128(to_dev(A))
    b8, sb = fq.quant_w_128x128(to_dev(B))
    C_full = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_ws(a8, sa, b8, sb, C_full, fq.BSCALE_BLOCK128, fq.workspace())
    kp = 4096                                   # the prefix the pages quote
    C_pre = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fq.fp8q_gemm_ws(a8[:, :kp].contiguous(), sa[:kp // 128].contiguous(),
                    b8[:, :kp].contiguous(), sb[:, :kp // 128].contiguous(), C_pre,
                    fq.BSCALE_BLOCK128, fq.workspace())
    assert fq.fp8q_get_device_status() == 0
    # 32 x 32 sampled outputs (tile corners among them), quantized by the oracle
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.integers(0, M, 28)]))[:32]
    cols = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 28)]))[:32]
    A8o, sAo = oracle.quant_1x128(A[rows])
    B8o, sBo = oracle.quant_128x128(B)
    B8c = np.ascontiguousarray(B8o[cols])
    sBc = np.ascontiguousarray(sBo[cols // 128].T)          # per-column scales [Kb][n]
    rel = {}
    for kmax, Cg in ((kp, C_pre), (K, C_full)):
        ref = oracle.gemm_prefix(A8o, sAo, B8c, sBc, kmax, bmode=1)
        got = cpu(Cg)[np.ix_(rows, cols)].astype(np.float64)
        rel["gpu", kmax] = float(np.max(np.abs(got - ref) / ref))
        emu = oracle.gemm_trunc_emu(A8o, sAo, B8c, sBc, kmax=kmax, chunk=4, mbits=13, bmode=1)
        rel["emu", kmax] = float(np.max(np.abs(emu - ref) / ref))
    print("\naccumulation stress, all-positive, max relative error over 32x32 outputs: "
          "GPU (promotion every 128) K=4096 %.3g, K=16384 %.3g; emulator without promotion "
          "K=4096 %.3g, K=16384 %.3g" % (rel["gpu", kp], rel["gpu", K], rel["emu", kp],
                                         rel["emu", K]))
    assert rel["gpu", kp] <= 1e-5 and rel["gpu", K] <= 1e-5
    assert 0.01 <= rel["emu", kp] <= 0.04
    assert rel["emu", K] > rel["emu", kp]        # the error grows with the reduction length
