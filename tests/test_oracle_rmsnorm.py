"""Pins of the oracle's RMSNorm and fused RMSNorm + 1x128 cast (woojincopolymer
post, para. 3) against facts that do not restate its formula:

- with w = 1 and eps = 0 every row of y has sum of squares exactly K (a mean
  taken as a sum, a missing square root or a misplaced eps breaks it);
- scale invariance: RMSNorm(a x) = RMSNorm(x) for a > 0 when eps = 0;
- one-hot row v e_j, w = 1, eps = 0: y_j = sign(v) sqrt(K), the rest 0;
- constant row c with eps: y = c w / sqrt(c^2 + eps) (closed form);
- the weight multiplies channel k only (a transposed or missing weight fails);
- with w = 1, eps = 0 and rows whose RMS is a power of two, y = x / rms is an
  exact scaling, so the fused cast equals the plain 1x128 quantizer applied to
  the row divided by that power of two, bit for bit."""
import numpy as np

import oracle


def test_sum_of_squares_is_K():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((16, 1024)).astype(np.float32) * 3.0
    y = oracle.rmsnorm_f64(x, np.ones(1024, np.float32), 0.0)
    assert np.allclose((y * y).sum(axis=1), 1024.0, rtol=1e-12)


def test_scale_invariance():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 512)).astype(np.float32)
    w = rng.standard_normal(512).astype(np.float32)
    y1 = oracle.rmsnorm_f64(x, w, 0.0)
    y2 = oracle.rmsnorm_f64(x * np.float32(64.0), w, 0.0)     # exact scaling by 2^6
    assert np.allclose(y1, y2, rtol=1e-13, atol=0)


def test_one_hot_row():
    K = 896
    x = np.zeros((2, K), np.float32)
    x[0, 17] = -3.5
    x[1, 500] = 1e-3
    y = oracle.rmsnorm_f64(x, np.ones(K, np.float32), 0.0)
    want = np.zeros((2, K))
    want[0, 17] = -np.sqrt(K)
    want[1, 500] = np.sqrt(K)
    assert np.allclose(y, want, rtol=1e-13, atol=1e-300)


def test_constant_row_with_eps():
    K, c, eps = 256, 0.25, 1e-2
    x = np.full((1, K), c, np.float32)
    w = np.linspace(-2.0, 2.0, K).astype(np.float32)
    y = oracle.rmsnorm_f64(x, w, eps)
    want = c * w.astype(np.float64) / np.sqrt(c * c + eps)
    assert np.allclose(y[0], want, rtol=1e-13, atol=1e-15)


def test_weight_is_per_channel():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 384)).astype(np.float32)
    w = np.zeros(384, np.float32)
    w[[5, 200]] = [2.0, -1.0]
    y = oracle.rmsnorm_f64(x, w, 1e-6)
    y1 = oracle.rmsnorm_f64(x, np.ones(384, np.float32), 1e-6)
    assert np.all(y[:, [i for i in range(384) if i not in (5, 200)]] == 0.0)
    assert np.allclose(y[:, 5], 2.0 * y1[:, 5], rtol=1e-14)
    assert np.allclose(y[:, 200], -y1[:, 200], rtol=1e-14)


def test_power_of_two_rms_reduces_to_plain_quantizer():
    # rows of +-a with a a power of two: rms = a exactly, y = x / a exactly
    rng = np.random.default_rng(4)
    K = 512
    signs = np.where(rng.random((6, K)) < 0.5, -1.0, 1.0).astype(np.float32)
    a = (2.0 ** np.arange(-3, 3)).astype(np.float32)[:, None]
    x = signs * a
    q, s, y = oracle.rmsnorm_quant_1x128(x, np.ones(K, np.float32), 0.0)
    q0, s0 = oracle.quant_1x128(signs)
    assert np.array_equal(q, q0)
    assert np.array_equal(s.view(np.uint32), s0.view(np.uint32))
