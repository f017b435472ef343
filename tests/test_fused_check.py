"""The interval check used for the fused RMSNorm / SwiGLU casts
(helpers.check_fused_1x128) must reject what it is meant to reject.  It is
fed the oracle's own result, which passes, and then that result with one
planted mistake: a code moved by one E4M3 step away from a rounding
boundary, a scale off by 1e-4, or a whole tile's codes shifted.  Each
planted mistake must fail.  Runs on the CPU only."""
import numpy as np
import pytest

from helpers import check_fused_1x128, exact_scaled_1x128


def case(oracle):
    rng = np.random.default_rng(21)
    g = (rng.standard_normal((8, 256)) * 2).astype(np.float32)
    u = rng.standard_normal((8, 256)).astype(np.float32)
    q, s, h = oracle.swiglu_quant_1x128(g, u)
    return q, s, h


def test_oracle_result_passes(oracle):
    q, s, h = case(oracle)
    check_fused_1x128(oracle, q, s, h, q, s, 6e-6, 3e-6, "self")


def test_one_code_moved_one_step_fails(oracle):
    q, s, h = case(oracle)
    y = exact_scaled_1x128(h)
    # an element far from a rounding boundary: |y| in the middle of [1, 448)
    dec = oracle.e4m3_decode(q)
    far = np.argwhere((np.abs(y) > 1.0) & (np.abs(y) < 400.0) &
                      (np.abs(np.abs(y) - np.abs(dec)) < 0.05 * np.abs(dec)))
    i = tuple(far[0])
    bad = q.copy()
    bad[i] = bad[i] + 1 if (bad[i] & 0x7F) < 0x7E else bad[i] - 1
    with pytest.raises(AssertionError):
        check_fused_1x128(oracle, bad, s, h, q, s, 6e-6, 3e-6, "moved code")


def test_scale_off_fails(oracle):
    q, s, h = case(oracle)
    bad = s.copy()
    bad[1, 3] *= np.float32(1.0001)
    with pytest.raises(AssertionError):
        check_fused_1x128(oracle, q, bad, h, q, s, 6e-6, 3e-6, "scale")


def test_shifted_tile_fails(oracle):
    q, s, h = case(oracle)
    bad = q.copy()
    mag = bad[2, 128:256] & 0x7F
    bad[2, 128:256] = np.where(mag < 0x7E, bad[2, 128:256] + 1, bad[2, 128:256])
    with pytest.raises(AssertionError):
        check_fused_1x128(oracle, bad, s, h, q, s, 6e-6, 3e-6, "tile")
