"""Pins of the oracle's SwiGLU and fused SwiGLU + 1x128 cast (woojincopolymer
post, paras. 3-4) against facts that do not restate its formula:

- silu(g) - silu(-g) = g (since sigmoid(g) + sigmoid(-g) = 1): a dropped or
  sign-flipped exponent breaks it;
- sigmoid(ln 3) = 3/4, so SwiGLU(ln 3, u) = (3/4) u ln 3;
- an independent route, sigmoid(g) = (1 + tanh(g/2)) / 2 via math.tanh;
- for g >= 40 and u = 1, SwiGLU(g, 1) rounds to g itself, so the fused cast
  must equal the (separately pinned) plain 1x128 quantizer bit for bit;
- zeros: SwiGLU(0, u) = SwiGLU(g, 0) = 0 and the tile scale is 1."""
import math

import numpy as np

import fp8q_inputs as fi
import oracle


def test_silu_odd_part_identity():
    g = np.linspace(-30.0, 30.0, 601, dtype=np.float32)
    one = np.ones_like(g)
    d = oracle.swiglu_f64(g, one) - oracle.swiglu_f64(-g, one)
    assert np.allclose(d, g.astype(np.float64), rtol=1e-14, atol=1e-14)


def test_sigmoid_of_log3():
    g = np.array([math.log(3.0)], np.float32)
    u = np.array([-2.5], np.float32)
    want = 0.75 * float(g[0]) * (-2.5)
    # g is ln 3 rounded to FP32; sigmoid(g) = 3/4 to first order in that rounding
    got = oracle.swiglu_f64(g, u)[0]
    sig = 1.0 / (1.0 + math.exp(-float(g[0])))
    assert abs(sig - 0.75) < 1e-7
    assert abs(got - want) <= 1e-6 * abs(want)


def test_against_tanh_route():
    rng = np.random.default_rng(5)
    g = rng.uniform(-8.0, 8.0, 4096).astype(np.float32)
    u = rng.standard_normal(4096).astype(np.float32)
    h = oracle.swiglu_f64(g, u)
    for i in range(0, 4096, 7):
        gi, ui = float(g[i]), float(u[i])
        ref = gi * ui * 0.5 * (1.0 + math.tanh(0.5 * gi))
        assert abs(h[i] - ref) <= 1e-13 * max(abs(ref), 1e-300), (gi, ui, h[i], ref)


def test_large_gate_reduces_to_plain_quantizer():
    rng = np.random.default_rng(6)
    g = rng.uniform(40.0, 400.0, (64, 512)).astype(np.float32)
    g = fi.to_bf16_bits(g)                      # BF16 inputs, as the fused kernel takes them
    u = fi.to_bf16_bits(np.ones((64, 512), np.float32))
    q, s, h = oracle.swiglu_quant_1x128(g, u)
    q0, s0 = oracle.quant_1x128(g)
    assert np.array_equal(q, q0)
    assert np.array_equal(s.view(np.uint32), s0.view(np.uint32))


def test_zeros():
    g = np.zeros((3, 256), np.float32)
    u = np.random.default_rng(7).standard_normal((3, 256)).astype(np.float32)
    q, s, h = oracle.swiglu_quant_1x128(g, u)
    assert np.all(h == 0.0)
    assert np.all(s == 1.0)
    assert np.all((q == 0x00) | (q == 0x80))
    q, s, h = oracle.swiglu_quant_1x128(u, np.zeros_like(u))
    assert np.all(h == 0.0) and np.all(s == 1.0)


def test_very_negative_gate_goes_to_signed_zero():
    g = np.full((1, 128), -800.0, np.float32)
    u = np.where(np.arange(128) % 2 == 0, 1.0, -1.0).astype(np.float32)[None, :]
    h = oracle.swiglu_f64(g, u)
    assert np.all(h == 0.0)
    # silu(-800) is -0 in FP64: the product's sign is -sign(u)
    assert np.array_equal(np.signbit(h[0]), u[0] > 0)
