"""Pins of the oracle's E4M3 codec (CPU only).

The pins do not come from the oracle itself: special values fixed by the E4M3
definition, torch's own float8_e4m3fn decoder and cast (an independent
implementation; its cast does not saturate, so it is used only in range),
and structural properties (round trip, ties to the even code, saturation).
"""
import math

import numpy as np
import torch


def torch_decode(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy())
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(vals):
    t = torch.from_numpy(np.asarray(vals, dtype=np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


ALL = np.arange(256, dtype=np.uint8)
NAN_CODES = {0x7F, 0xFF}


def test_decode_all_256_against_torch(oracle):
    ours = oracle.e4m3_decode(ALL)
    ref = torch_decode(ALL)
    for b in range(256):
        if b in NAN_CODES:
            assert math.isnan(ours[b])
        else:
            assert ours[b] == ref[b], hex(b)
            assert math.copysign(1.0, ours[b]) == math.copysign(1.0, ref[b]), hex(b)


def test_decode_special_values(oracle):
    d = oracle.e4m3_decode(ALL)
    assert d[0x7E] == 448.0                      # max finite
    assert d[0xFE] == -448.0
    assert d[0x01] == 2.0 ** -9                  # min subnormal
    assert d[0x07] == 7 * 2.0 ** -9              # max subnormal
    assert d[0x08] == 2.0 ** -6                  # min normal
    assert d[0x38] == 1.0
    assert d[0x00] == 0.0 and math.copysign(1, d[0x00]) == 1
    assert d[0x80] == 0.0 and math.copysign(1, d[0x80]) == -1
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)              # codes 0x00..0x7E increase strictly


def test_round_trip_every_finite_code(oracle):
    codes = np.array([b for b in range(256) if b not in NAN_CODES], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_tie_to_even_code(oracle):
    d = oracle.e4m3_decode(ALL)
    for c in range(0x7E):
        mid = np.float32(0.5 * (d[c] + d[c + 1]))
        assert float(mid) == 0.5 * (d[c] + d[c + 1])      # exact in FP32
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == even, hex(c)
        assert oracle.e4m3_encode([-mid])[0] == (0x80 | even), hex(c)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        assert oracle.e4m3_encode([below])[0] == c
        assert oracle.e4m3_encode([above])[0] == c + 1


def test_saturation_nan_and_underflow(oracle):
    enc = lambda v: int(oracle.e4m3_encode([v])[0])
    assert enc(448.0) == 0x7E
    assert enc(464.0) == 0x7E
    assert enc(470.0) == 0x7E
    assert enc(1e6) == 0x7E
    assert enc(float("inf")) == 0x7E
    assert enc(-float("inf")) == 0xFE
    assert enc(-1e30) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(2.0 ** -10) == 0x00               # tie between 0 and 2^-9 -> even (0)
    assert enc(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01
    assert enc(-(2.0 ** -10)) == 0x80            # sign of zero kept
    assert enc(-0.0) == 0x80
    assert enc(1e-40) == 0x00                    # FP32 subnormal input


def test_encode_matches_torch_in_range(oracle):
    rng = np.random.default_rng(1234)
    n = 200_000
    mag = np.exp2(rng.uniform(-14.0, math.log2(464.0), n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    v = mag * sign
    v = v[np.abs(v) <= 464.0]
    assert np.array_equal(oracle.e4m3_encode(v), torch_encode(v))


def test_encode_matches_nearest_by_distance(oracle):
    """Nearest-value property checked by plain distances on random inputs."""
    rng = np.random.default_rng(7)
    d = oracle.e4m3_decode(ALL)[:0x7F]
    v = rng.uniform(0, 448, 20_000).astype(np.float32)
    q = oracle.e4m3_encode(v)
    dist_chosen = np.abs(d[q] - v.astype(np.float64))
    dist_best = np.min(np.abs(d[None, :] - v.astype(np.float64)[:, None]), axis=1)
    assert np.array_equal(dist_chosen, dist_best)
