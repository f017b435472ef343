"""GPU parity of the GEMM that quantizes its BF16 activations itself
(fp8q_gemm_quant_a; woojincopolymer post, para. 4: the FP8 cast fused with
the global-to-shared transfer).  Its definition is the composition of two
pinned oracle steps: A8, sA = quant_1x128(A), then the block-scaled GEMM.  So:
  * the emitted A8 bytes and sA scales are bit-exact against the oracle's
    1x128 quantizer (every element for small shapes, sampled rows of the
    forward workload), including the scale rule's edge cases;
  * C is within the GEMM tolerance of the oracle GEMM of those operands
    (1e-5 sum_k |a_k b_k|, plus one BF16 ulp for BF16 output).
Shapes cover several tiles per CTA, stream-K cuts and whole tiles."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import Guarded, assert_gemm_close, cpu, to_dev
from test_gpu_gemm import check_sampled, corner_and_random
from test_gpu_quant import assert_bytes_equal, assert_scales_equal, special_tile_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def run_fused(fq, A_bits, B8, sB, out, emit=True, stream_k=True):
    M, K = A_bits.shape
    N = B8.shape[0]
    C = Guarded((M, N), out, fill=float("nan"))
    A8 = Guarded((M, K), torch.uint8) if emit else None
    sA = Guarded((K // 128, M), torch.float32) if emit else None
    fq.fp8q_gemm_quant_a(to_dev(A_bits), to_dev(B8), to_dev(sB), C.t, A8.t if emit else None,
                         sA.t if emit else None, fq.workspace() if stream_k else None)
    assert fq.fp8q_get_device_status() == 0
    C.check("C")
    if emit:
        A8.check("A8_out")
        sA.check("sA_out")
    return C.t, (A8.t if emit else None), (sA.t if emit else None)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [
    (128, 256, 128),      # one tile, one K block
    (256, 256, 1024),
    (384, 512, 640),      # 3 x 2 tiles, 5 K blocks
    (1024, 768, 1280),    # 8 x 3 tiles, 10 K blocks
])
@pytest.mark.parametrize("stream_k", [True, False])
def test_fused_quant_gemm_small(fq, oracle, out, M, N, K, stream_k):
    A = special_tile_input(M, K, True, seed=M + N + K)          # BF16 bits, edge-case tiles
    W = fi.gaussian((N, K), fi.rng_for(M + N, 1), 0.02, bf16=False)
    B8, sB = oracle.quant_128x128(W)
    C, A8, sA = run_fused(fq, A, B8, sB, out, emit=True, stream_k=stream_k)
    A8o, sAo = oracle.quant_1x128(A)
    assert_bytes_equal(cpu(A8), A8o, "A8_out")
    assert_scales_equal(cpu(sA), sAo, "sA_out")
    Cref, Cabs = oracle.gemm(A8o, sAo, B8, sB)
    assert_gemm_close(cpu(C), Cref, Cabs, out == torch.bfloat16, "fused quant + GEMM")


def test_fused_quant_gemm_without_emit_matches_two_step(fq, oracle):
    """Without A8_out/sA_out the result is the same GEMM: compared with the
    two-step path (fp8q_quant_act_1x128, then fp8q_gemm_ws) within the
    tolerance, on many tiles per CTA."""
    M, N, K = 4096, 1536, 384                                    # 32 x 6 = 192 tiles
    A = fi.gaussian((M, K), fi.rng_for(61, 0), 1.0, 0.001, 100.0)
    W = fi.gaussian((N, K), fi.rng_for(61, 1), 0.02, bf16=False)
    B8, sB = oracle.quant_128x128(W)
    C, _, _ = run_fused(fq, A, B8, sB, torch.bfloat16, emit=False)
    a8, sa = fq.quant_act_1x128(to_dev(A))
    C2 = torch.empty_like(C)
    fq.fp8q_gemm_ws(a8, sa, to_dev(B8), to_dev(sB), C2, fq.BSCALE_BLOCK128, fq.workspace())
    rng = np.random.default_rng(61)
    rows = corner_and_random(M, 48, rng)
    cols = np.arange(N)
    A8o, sAo = oracle.quant_1x128(A[rows])
    B8c = np.ascontiguousarray(B8[cols])
    sBc = np.ascontiguousarray(sB[cols // 128].T)
    check_sampled(cpu(C), rows, cols, A8o, sAo, B8c, sBc, 1, True, "fused (no emit)", rng)
    check_sampled(cpu(C2), rows, cols, A8o, sAo, B8c, sBc, 1, True, "two-step", rng)


def test_fused_argument_checks(fq, oracle):
    A = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    B8 = torch.zeros(384, 256, dtype=torch.uint8, device="cuda")     # N % 256 != 0
    sB = torch.zeros(3, 2, dtype=torch.float32, device="cuda")
    C = torch.zeros(256, 384, dtype=torch.float32, device="cuda")
    with pytest.raises(fq.Fp8qError) as e:
        fq.fp8q_gemm_quant_a(A, B8, sB, C)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        fq.fp8q_gemm_quant_a(A, B8, sB, C, A8_out=torch.zeros(256, 256, dtype=torch.uint8,
                                                                 device="cuda"))
    assert torch.count_nonzero(C).item() == 0                      # nothing launched


@pytest.mark.slow
def test_fused_quant_gemm_forward_workload(fq, oracle):
    """The forward workload (A[4096][7168] BF16 with outliers, W[2048][7168]):
    emitted tiles bit-exact on sampled rows, C within tolerance on sampled
    entries (tile corners and random)."""
    d = fi.make("forward")
    w8, sw = fq.quant_w_128x128(to_dev(d["W"]))
    C, A8, sA = fq.gemm_quant_a(to_dev(d["A"]), w8, sw, out_dtype=torch.bfloat16)
    assert fq.fp8q_get_device_status() == 0
    rng = np.random.default_rng(62)
    rows = corner_and_random(4096, 32, rng)
    cols = corner_and_random(2048, 32, rng)
    A8o, sAo = oracle.quant_1x128(d["A"][rows])
    assert_bytes_equal(cpu(A8)[rows], A8o, "A8_out rows")
    assert_scales_equal(cpu(sA)[:, rows], sAo, "sA_out rows")
    B8o, sBo = oracle.quant_128x128(d["W"])
    B8c = np.ascontiguousarray(B8o[cols])
    sBc = np.ascontiguousarray(sBo[cols // 128].T)
    check_sampled(cpu(C), rows, cols, A8o, sAo, B8c, sBc, 1, True, "fused forward", rng)
