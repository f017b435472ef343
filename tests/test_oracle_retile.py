"""Pins of the oracle's backward regrouping (stored 1x128 FP8 tiles ->
128x1 tiles, "Six Reasons Deepseek Ai Is A Waste Of Time", paragraph 3).

The main pin is an identity that does not use the regrouping's own code: when
every 1x128 tile of x is a power of two times E4M3 values, with the value 448
times that power present, the forward quantization is exact, so regrouping its
tiles must give exactly the (separately pinned) 128x1 quantization of x.  A
wrong scale index, a transposed operand or a dropped dequantization fails it.
"""
import numpy as np

import fp8q_inputs as fi

E4M3_POS = None


def e4m3_values(oracle):
    global E4M3_POS
    if E4M3_POS is None:
        v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))      # 0x00 .. 0x7E
        E4M3_POS = v[np.isfinite(v)]
    return E4M3_POS


def exact_tiles(oracle, T, C, seed):
    """x[T][C] whose 1x128 tiles quantize exactly: values = +-E4M3 * 2^e(tile),
    one element of each tile equal to +-448 * 2^e(tile)."""
    rng = np.random.default_rng(seed)
    vals = e4m3_values(oracle)
    x = np.empty((T, C), np.float64)
    for t in range(T):
        for g in range(0, C, 128):
            w = min(128, C - g)
            e = int(rng.integers(-12, 6))
            tile = rng.choice(vals, w) * rng.choice([-1.0, 1.0], w)
            tile[int(rng.integers(0, w))] = 448.0 * rng.choice([-1.0, 1.0])
            x[t, g:g + w] = tile * 2.0 ** e
    return x.astype(np.float32)


def test_exact_tiles_regroup_to_the_128x1_quantization(oracle):
    T, C = 384, 256
    x = exact_tiles(oracle, T, C, seed=1)
    q, s = oracle.quant_1x128(x)
    assert np.array_equal(oracle.dequant_1x128(q, s), x.astype(np.float64))   # premise: exact
    qT, sT = oracle.retile_1x128_to_128x1(q, s)
    qT_ref, sT_ref = oracle.quant_128x1(x)
    assert np.array_equal(qT, qT_ref)
    assert np.array_equal(sT.view(np.uint32), sT_ref.view(np.uint32))


def test_one_hot(oracle):
    T, C = 256, 128
    q = np.zeros((T, C), np.uint8)
    s = np.ones((1, T), np.float32)
    q[200, 37] = 0xD6                    # -(1.75 * 2^3) = -14
    s[0, 200] = np.float32(0.375)
    qT, sT = oracle.retile_1x128_to_128x1(q, s)
    want = np.zeros((C, T), np.uint8)
    want[37, 200] = 0xFE                 # -448: the tile's only nonzero maps to -max
    assert np.array_equal(qT, want)
    assert sT[1, 37] == np.float32(np.float32(14.0 * 0.375) / np.float32(448.0))
    assert np.all(np.delete(sT.ravel(), 1 * C + 37) == 1.0)    # empty tiles keep scale 1


def test_zero_input(oracle):
    q = np.zeros((128, 256), np.uint8)
    s = np.full((2, 128), 3.0, np.float32)
    qT, sT = oracle.retile_1x128_to_128x1(q, s)
    assert not qT.any() and np.all(sT == 1.0)


def test_two_stage_error_bound(oracle):
    """Each quantization moves an element by at most 2^-4 of itself plus
    2^-10 of its tile's scale (E4M3 has 3 mantissa bits, subnormal step
    2^-9); two of them, applied in turn, bound the regrouped value."""
    T, C = 256, 384
    x = fi.gaussian((T, C), fi.rng_for(4, 0), 1.0, 0.01, 100.0, bf16=False)
    q, s = oracle.quant_1x128(x)
    x1 = oracle.dequant_1x128(q, s)
    qT, sT = oracle.retile_1x128_to_128x1(q, s)
    x2 = oracle.dequant_1x128(qT, sT).T                        # back to [T][C]
    s1 = np.repeat(s.T.astype(np.float64), 128, axis=1)[:, :C]
    s2 = np.repeat(sT.astype(np.float64), 128, axis=0)[:T, :]
    e = 1 + 2.0 ** -20
    assert np.all(np.abs(x1 - x) <= (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s1) * e)
    assert np.all(np.abs(x2 - x1) <= (2.0 ** -4 * np.abs(x1) + 2.0 ** -10 * s2) * e)


def test_ragged_tokens(oracle):
    """T not a multiple of 128: the last token group is partial."""
    x = exact_tiles(oracle, 200, 128, seed=5)
    q, s = oracle.quant_1x128(x)
    qT, sT = oracle.retile_1x128_to_128x1(q, s)
    qT_ref, sT_ref = oracle.quant_128x1(x)
    assert np.array_equal(qT, qT_ref) and np.array_equal(sT, sT_ref)
