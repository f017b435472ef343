"""GPU parity of the fused SwiGLU + 1x128 FP8 cast against the CPU oracle.

Tolerance, from the arithmetic: the kernel evaluates h = g u / (1 + e^-g) in
FP32 -- e^-g by CUDA's expf (documented to within 2 ulp), then an add, a
division and a multiplication, each correctly rounded -- so h_gpu = h (1 + d)
with |d| below about 5 ulp (3e-7); a tile's amax, hence its scale and
inverse, carries the same bound.  The test asks for ten times that:
  * scales within 3e-6 relative of the oracle's;
  * every code the round-to-nearest-even E4M3 encoding of some value within
    6e-6 relative of the exact scaled value h * inv (an interval check: at a
    rounding boundary either neighbour passes, anywhere else only one code);
  * at least 99.9 % of the codes identical to the oracle's, so the interval
    cannot hide a systematic error.
Where the FP32 evaluation is exact (large gates, zero gates) the comparison
is bit for bit."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import check_fused_1x128, cpu, to_dev

pytestmark = pytest.mark.gpu

H_REL = 6e-6
S_REL = 3e-6


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def check(oracle, q_gpu, s_gpu, g, u, what):
    q_o, s_o, h = oracle.swiglu_quant_1x128(g, u)
    check_fused_1x128(oracle, q_gpu, s_gpu, h, q_o, s_o, H_REL, S_REL, what)
    return q_o, s_o


def inputs(M, I, bf16, seed):
    g = fi.gaussian((M, I), fi.rng_for(seed, 0), 2.0, 0.001, 100.0, bf16=False)
    u = fi.gaussian((M, I), fi.rng_for(seed, 1), 1.0, 0.001, 100.0, bf16=False)
    if M >= 4 and I >= 256:
        g[0, :128] = 0.0                            # zero gate: h = +-0, scale 1
        g[1, 128:256] = -200.0                      # e^-g overflows: h = -0 * u
        g[1, 130] = 3.0                             # ... except one element
        g[2, :128] = np.float32(1e-30)              # tiny gate: h ~ g u / 2
        u[3, :128] = 0.0
    if bf16:
        return fi.to_bf16_bits(g), fi.to_bf16_bits(u)
    return g, u


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("M,I", [(1, 128), (37, 256), (64, 384), (130, 1024)])
def test_swiglu_quant_small(fq, oracle, bf16, M, I):
    g, u = inputs(M, I, bf16, seed=M * 7 + I)
    q, s = fq.swiglu_quant_1x128(to_dev(g), to_dev(u))
    check(oracle, cpu(q), cpu(s), g, u, "M=%d I=%d" % (M, I))


def test_swiglu_quant_strided_halves(fq, oracle):
    """gate and up as the two halves of one [M][2I] tensor (row stride 2I)."""
    M, I = 200, 512
    g, u = inputs(M, I, True, seed=3)
    gu = to_dev(np.concatenate([g, u], axis=1))
    q1, s1 = fq.swiglu_quant_1x128(gu[:, :I], gu[:, I:])
    q2, s2 = fq.swiglu_quant_1x128(to_dev(g), to_dev(u))
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    check(oracle, cpu(q1), cpu(s1), g, u, "strided")


def test_swiglu_quant_large_gate_is_plain_quantizer(fq, oracle):
    """g >= 40, u = 1: e^-g < 5e-18 vanishes against 1 in FP32, h = g exactly,
    so the fused kernel equals the plain 1x128 quantizer (and the oracle) bit
    for bit."""
    rng = np.random.default_rng(11)
    g = fi.to_bf16_bits(rng.uniform(40.0, 400.0, (96, 640)).astype(np.float32)
                        * np.where(rng.random((96, 640)) < 0.5, 1.0, 1.0).astype(np.float32))
    u = fi.to_bf16_bits(np.ones((96, 640), np.float32))
    q, s = fq.swiglu_quant_1x128(to_dev(g), to_dev(u))
    q0, s0 = fq.quant_act_1x128(to_dev(g))
    assert torch.equal(q, q0) and torch.equal(s, s0)
    qo, so, _ = oracle.swiglu_quant_1x128(g, u)
    assert np.array_equal(cpu(q), qo) and np.array_equal(cpu(s).view(np.uint32), so.view(np.uint32))


def test_swiglu_quant_zero_gate_bit_exact(fq, oracle):
    g = np.zeros((32, 256), np.float32)
    u = np.random.default_rng(12).standard_normal((32, 256)).astype(np.float32)
    q, s = fq.swiglu_quant_1x128(to_dev(g), to_dev(u))
    qo, so, _ = oracle.swiglu_quant_1x128(g, u)
    assert np.array_equal(cpu(q), qo)                 # +-0 with the sign of u
    assert np.all(cpu(s) == 1.0)


def test_swiglu_quant_argument_errors(fq):
    g = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fq.swiglu_quant_1x128(g, g[:, :128])
    with pytest.raises(fq.Fp8qError) as e:
        fq.swiglu_quant_1x128(g[:, :200], g[:, 56:])
    assert e.value.status == 2                        # I not a multiple of 128


@pytest.mark.slow
def test_swiglu_quant_mlp_workload(fq, oracle):
    """The bench's down-projection input: gate_up[4096][2 x 2048], sampled rows."""
    d = fi.make("mlp_down")
    gu = d["gate_up"]
    I = gu.shape[1] // 2
    dgu = to_dev(gu)
    q, s = fq.swiglu_quant_1x128(dgu[:, :I], dgu[:, I:])
    qg, sg = cpu(q), cpu(s)
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([[0, gu.shape[0] - 1], rng.integers(0, gu.shape[0], 48)]))
    check(oracle, qg[rows], sg[:, rows], gu[rows, :I], gu[rows, I:], "mlp_down rows")
