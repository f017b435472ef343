"""GPU parity of the fused RMSNorm + 1x128 FP8 cast against the CPU oracle.

Tolerance, from the arithmetic: the kernel sums the row's squares in FP32 --
16 fused multiply-adds per thread, then two five-level shuffle trees -- so
the mean carries at most about 26 roundings (1.6e-6 relative); the reciprocal
square root is correctly rounded and y = (x r) w adds two more roundings.
y is thus within about 2e-6 relative of the exact value, and so are a tile's
amax, scale and inverse.  The test asks for ten times that: scales within
1e-5 relative, every code the RNE E4M3 encoding of a value within 2e-5
relative of the exact scaled value, at least 99.9 % of the codes identical to
the oracle's (tests/helpers.check_fused_1x128)."""
import numpy as np
import pytest
import torch

import fp8q_inputs as fi
from helpers import check_fused_1x128, cpu, to_dev

pytestmark = pytest.mark.gpu

H_REL = 2e-5
S_REL = 1e-5
EPS = 1e-6


@pytest.fixture(scope="module")
def fq():
    import fp8_fine_grained_21_b300 as m

    m.load()
    return m


def inputs(M, K, bf16, seed):
    x = fi.gaussian((M, K), fi.rng_for(seed, 0), 1.0, 0.001, 100.0, bf16=False)
    w = (1.0 + 0.1 * fi.rng_for(seed, 1).standard_normal(K)).astype(np.float32)
    if M >= 4:
        x[0] = 0.0                                   # zero row: y = 0, scale 1
        x[1, :] = 0.0
        x[1, 300 % K] = -7.0                         # one-hot row
        x[2] *= np.float32(1e-3)                     # small row (eps matters a little)
        x[3, :128] = 0.0                             # one zero tile in a normal row
    if bf16:
        return fi.to_bf16_bits(x), fi.to_bf16_bits(w)
    return x, w


def check(oracle, q, s, x, w, what):
    q_o, s_o, y = oracle.rmsnorm_quant_1x128(x, w, EPS)
    check_fused_1x128(oracle, q, s, y, q_o, s_o, H_REL, S_REL, what)


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (64, 1024), (130, 7168), (5, 16384)])
def test_rmsnorm_quant(fq, oracle, bf16, M, K):
    x, w = inputs(M, K, bf16, seed=M * 3 + K)
    q, s = fq.rmsnorm_quant_1x128(to_dev(x), to_dev(w), EPS)
    check(oracle, cpu(q), cpu(s), x, w, "M=%d K=%d" % (M, K))


def test_rmsnorm_quant_argument_errors(fq):
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fq.Fp8qError) as e:
        fq.rmsnorm_quant_1x128(x, w, 0.0)
    assert e.value.status == 1                        # eps must be > 0
    big = torch.zeros((2, 16384 + 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fq.Fp8qError) as e:
        fq.rmsnorm_quant_1x128(big, torch.ones(16384 + 128, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 2                        # K above 16384
    with pytest.raises(ValueError):
        fq.rmsnorm_quant_1x128(x, w[:128])


@pytest.mark.slow
def test_rmsnorm_quant_forward_workload(fq, oracle):
    """The bench's normalized forward input: x[4096][7168], sampled rows."""
    d = fi.make("forward_norm")
    x, w = d["X"], d["g"]
    q, s = fq.rmsnorm_quant_1x128(to_dev(x), to_dev(w), EPS)
    qg, sg = cpu(q), cpu(s)
    rng = np.random.default_rng(17)
    rows = np.unique(np.concatenate([[0, x.shape[0] - 1], rng.integers(0, x.shape[0], 48)]))
    check(oracle, qg[rows], sg[:, rows], x[rows], w, "forward_norm rows")
