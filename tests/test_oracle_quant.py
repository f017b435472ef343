"""Pins of the oracle's online quantizers (CPU only).

Hand-worked golden tile, closed forms (constant and one-hot tiles, power-of-two
maxima), the tile-max invariant, tile independence, the 128x1 / 1x128
transpose identity, ragged tails and the per-element error bound of a
round-to-nearest 3-bit-mantissa cast.
"""
import os

import numpy as np
import pytest

import fp8q_inputs as fi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_hand_tile():
    scale = None
    rows = []
    with open(os.path.join(GOLDEN, "quant_1x128_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "scale":
                scale = float.fromhex(parts[1])
            else:
                rows.append((int(parts[0]), float.fromhex(parts[1]), int(parts[2], 16)))
    return scale, rows


def test_hand_worked_tile(oracle):
    scale, rows = load_hand_tile()
    x = np.zeros((1, 128), np.float32)
    for i, v, _ in rows:
        x[0, i] = np.float32(v)
    q, s = oracle.quant_1x128(x)
    assert s.shape == (1, 1) and s[0, 0] == np.float32(scale)
    for i, _, b in rows:
        assert q[0, i] == b, (i, hex(q[0, i]), hex(b))
    rest = np.setdiff1d(np.arange(128), [r[0] for r in rows])
    assert np.all(q[0, rest] == 0)


def test_tile_scale_closed_forms(oracle):
    assert oracle.tile_scale(448.0) == (1.0, 1.0)
    assert oracle.tile_scale(896.0) == (2.0, 0.5)
    assert oracle.tile_scale(7.0) == (2.0 ** -6, 64.0)
    assert oracle.tile_scale(0.0) == (1.0, 1.0)          # all-zero tile
    s, inv = oracle.tile_scale(1e-38)                     # 448/amax overflows FP32
    assert inv == np.finfo(np.float32).max


@pytest.mark.parametrize("c", [1.0, -3.0, 0.125, 1000.0, -2.5e-3, 3.1415927])
def test_constant_tile(oracle, c):
    x = np.full((2, 256), np.float32(c))
    q, s = oracle.quant_1x128(x)
    code = 0x7E if c > 0 else 0xFE
    assert np.all(q == code)
    # s * 448 recovers |c| to within one FP32 rounding
    assert np.allclose(s.astype(np.float64) * 448.0, abs(c), rtol=2 ** -23, atol=0)


def test_one_hot_tiles(oracle):
    x = np.zeros((3, 128), np.float32)
    x[0, 5] = 448.0 * 4          # power of two times 448: s exactly 4
    x[1, 127] = -0.75
    x[2, 0] = 1e-3
    q, s = oracle.quant_1x128(x)
    assert s[0, 0] == 4.0
    assert q[0, 5] == 0x7E and q[1, 127] == 0xFE and q[2, 0] == 0x7E
    assert np.count_nonzero(q) == 3


def test_all_zero_and_negative_zero(oracle):
    x = np.zeros((1, 128), np.float32)
    x[0, 3] = -0.0
    q, s = oracle.quant_1x128(x)
    assert s[0, 0] == 1.0
    assert q[0, 3] == 0x80 and np.count_nonzero(q) == 1


def _tiles_1x128(x):
    M, K = x.shape
    return x.reshape(M, K // 128, 128)


def test_tile_max_maps_to_448(oracle):
    rng = fi.rng_for(11, 0)
    x = fi.gaussian((64, 1024), rng, 1.0, 0.01, 100.0, bf16=False)
    q, s = oracle.quant_1x128(x)
    xt, qt = _tiles_1x128(x), _tiles_1x128(q)
    idx = np.argmax(np.abs(xt), axis=2)
    sel = np.take_along_axis(qt, idx[..., None], axis=2)[..., 0]
    assert np.all((sel & 0x7F) == 0x7E)
    assert s.shape == (8, 64)


def test_tile_independence(oracle):
    rng = fi.rng_for(12, 0)
    x = fi.gaussian((16, 512), rng, bf16=False)
    q0, s0 = oracle.quant_1x128(x)
    y = x.copy()
    y[5, 256:384] *= np.float32(3.0)
    y[5, 300] = np.float32(77.0)
    q1, s1 = oracle.quant_1x128(y)
    changed_q = np.argwhere(q0 != q1)
    assert changed_q.size and np.all(changed_q[:, 0] == 5)
    assert np.all((changed_q[:, 1] >= 256) & (changed_q[:, 1] < 384))
    changed_s = np.argwhere(s0 != s1)
    assert changed_s.tolist() == [[2, 5]]


def test_128x1_is_1x128_of_transpose(oracle):
    rng = fi.rng_for(13, 0)
    x = fi.gaussian((384, 200), rng, 1.0, 0.01, 100.0, bf16=False)
    qT, sT = oracle.quant_128x1(x)
    q2, s2 = oracle.quant_1x128(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_128x128_block_structure(oracle):
    rng = fi.rng_for(14, 0)
    w = fi.gaussian((256, 384), rng, 0.02, bf16=False)
    q, s = oracle.quant_128x128(w)
    assert s.shape == (2, 3)
    for nb in range(2):
        for g in range(3):
            blk = w[nb * 128:(nb + 1) * 128, g * 128:(g + 1) * 128]
            qb = q[nb * 128:(nb + 1) * 128, g * 128:(g + 1) * 128]
            r, c = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert (qb[r, c] & 0x7F) == 0x7E
            # a block made of one repeated row quantizes like that row's 1x128 tile
    row = w[:1, :128]
    qr, sr = oracle.quant_1x128(row)
    qb, sb = oracle.quant_128x128(np.repeat(row, 128, axis=0))
    assert np.array_equal(qb, np.repeat(qr, 128, axis=0)) and sb[0, 0] == sr[0, 0]


def test_ragged_tails(oracle):
    rng = fi.rng_for(15, 0)
    x = fi.gaussian((5, 200), rng, bf16=False)
    q, s = oracle.quant_1x128(x)
    assert s.shape == (2, 5)
    tail = x[:, 128:]
    amax = np.max(np.abs(tail), axis=1)
    assert np.allclose(s[1].astype(np.float64) * 448.0, amax, rtol=2 ** -23)
    idx = np.argmax(np.abs(tail), axis=1)
    assert np.all((q[np.arange(5), 128 + idx] & 0x7F) == 0x7E)
    w = fi.gaussian((130, 129), rng, bf16=False)
    qw, sw = oracle.quant_128x128(w)
    assert sw.shape == (2, 2)
    assert np.allclose(sw[1, 1] * 448.0, np.max(np.abs(w[128:, 128:])), rtol=2 ** -23)


def test_error_bound(oracle):
    """|decode(q)*s - x| <= 2^-4 |x| + 2^-10 s (+ FP32 rounding slack):
    half a unit in the last place of a 3-bit mantissa, or half the subnormal
    spacing 2^-9 scaled back by s."""
    rng = fi.rng_for(16, 0)
    x = fi.gaussian((32, 1024), rng, 1.0, 0.01, 100.0, bf16=False)
    q, s = oracle.quant_1x128(x)
    sfull = np.repeat(s.T, 128, axis=1)
    deq = oracle.e4m3_decode(q) * sfull
    err = np.abs(deq - x.astype(np.float64))
    bound = 2.0 ** -4 * np.abs(x) * (1 + 2.0 ** -20) + 2.0 ** -10 * sfull * (1 + 2.0 ** -20)
    assert np.all(err <= bound)


def test_bf16_inputs_widen_exactly(oracle):
    rng = fi.rng_for(17, 0)
    xb = fi.gaussian((8, 256), rng)                  # uint16 BF16 bits
    q1, s1 = oracle.quant_1x128(xb)
    q2, s2 = oracle.quant_1x128(fi.bf16_bits_to_f32(xb))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
