"""Pins of the limited-precision accumulation emulator (CPU only).

Closed forms (no truncation reproduces the FP64 sum; a counter of ones stalls
where the retained bits run out) and the pages' one printed figure: without
promotion the maximum relative error at K = 4096 is close to 2% ("Six Reasons
Deepseek Ai Is A Waste Of Time", paragraph 2).  That figure comes with no
inputs or hardware model, so it pins the emulator's default knobs only to
order of magnitude (1%..4%) -- a loose pin.
"""
import numpy as np

import fp8q_inputs as fi


def test_no_truncation_is_fp64_sum(oracle):
    A = fi.uniform((16, 512), fi.rng_for(1, 0), bf16=False)
    B = fi.uniform((16, 512), fi.rng_for(1, 1), bf16=False)
    A8, sA = oracle.quant_1x128(A)
    B8, sB = oracle.quant_128x128(B)
    ref = oracle.gemm_prefix(A8, sA, B8, sB, 512)
    emu = oracle.gemm_trunc_emu(A8, sA, B8, sB, chunk=1, mbits=60)
    full, _ = oracle.gemm(A8, sA, B8, sB)
    assert np.array_equal(emu, ref) and np.array_equal(ref, full)


def test_counter_stalls_at_retained_bits(oracle):
    """Adding 1.0 repeatedly with 3 retained fraction bits: 16 + 1 = 17 needs 4
    fraction bits and truncates back to 16, so the sum sticks at 16."""
    K = 256
    A8 = np.full((1, K), 0x38, np.uint8)        # 1.0
    B8 = np.full((1, K), 0x38, np.uint8)
    sA = np.ones((2, 1), np.float32)
    sB = np.ones((1, 2), np.float32)
    assert oracle.gemm_trunc_emu(A8, sA, B8, sB, chunk=1, mbits=3)[0, 0] == 16.0
    # chunks of 4 exact products: steps of 4 fit 3 fraction bits up to 64 = 2^6,
    # where the unit in the last place becomes 8 and 64 + 4 truncates to 64
    assert oracle.gemm_trunc_emu(A8, sA, B8, sB, chunk=4, mbits=3)[0, 0] == 64.0
    # promotion every 128 elements restarts the limited accumulator: 2 x 16
    assert oracle.gemm_trunc_emu(A8, sA, B8, sB, chunk=1, mbits=3, promote=128)[0, 0] == 32.0
    # kmax limits the reduction to a prefix
    assert oracle.gemm_trunc_emu(A8, sA, B8, sB, kmax=10, chunk=1, mbits=3)[0, 0] == 10.0


def test_truncation_is_toward_zero(oracle):
    K = 128
    A8 = np.full((1, K), 0xB8, np.uint8)        # -1.0
    B8 = np.full((1, K), 0x38, np.uint8)
    sA = np.ones((1, 1), np.float32)
    sB = np.ones((1, 1), np.float32)
    assert oracle.gemm_trunc_emu(A8, sA, B8, sB, chunk=1, mbits=3)[0, 0] == -16.0


def test_two_percent_at_k4096_loose_pin(oracle):
    """All-positive U(0,1) operands (the accumulation-stress workload's
    positive variant), quantized 1x128 / 128x128, first 4096 elements of K."""
    M = N = 32
    A = fi.uniform((M, 4096), fi.rng_for(0, 0), 0.0, 1.0)
    B = fi.uniform((N, 4096), fi.rng_for(0, 1), 0.0, 1.0)
    A8, sA = oracle.quant_1x128(A)
    B8, sB = oracle.quant_128x128(B)
    ref = oracle.gemm_prefix(A8, sA, B8, sB, 4096)
    emu = oracle.gemm_trunc_emu(A8, sA, B8, sB, kmax=4096, chunk=4, mbits=13)
    rel = np.max(np.abs(emu - ref) / np.abs(ref))
    assert 0.01 <= rel <= 0.04, rel
    promoted = oracle.gemm_trunc_emu(A8, sA, B8, sB, kmax=4096, chunk=4, mbits=13, promote=128)
    rel_p = np.max(np.abs(promoted - ref) / np.abs(ref))
    assert rel_p < rel / 20, (rel_p, rel)


def test_prefix_sum_pins(oracle):
    """The FP64 prefix GEMM (the reference of the emulator's error) over the
    first kmax < K elements: (1) a closed form whose two 128-element scale
    groups carry different values, cut inside the second group, so that a
    wrong group index or a wrong cut shows; (2) the independent exact int64
    route applied to the K-truncated operands, for both B-scale layouts, at
    the K = 4096 prefix of a K = 16384 problem (the accumulation-stress
    shape's prefix)."""
    # (1) A = 7 in group 0 and 14 in group 1, B = 7/16: the scales 2^-6, 2^-5 and
    # 2^-10 are exact, every byte is 448, so every product and sum is exact
    K = 256
    A = np.concatenate([np.full((1, 128), 7.0), np.full((1, 128), 14.0)], axis=1).astype(np.float32)
    B = np.full((1, K), 0.4375, np.float32)
    A8, sA = oracle.quant_1x128(A)
    B8, sB = oracle.quant_1x128(B)
    for kmax, want in ((200, 128 * 7 * 0.4375 + 72 * 14 * 0.4375), (128, 392.0), (1, 3.0625),
                       (256, 1176.0)):
        got = oracle.gemm_prefix(A8, sA, B8, sB, kmax, bmode=1)[0, 0]
        assert got == want, (kmax, got, want)
    # (2) K-truncated operands through the exact integer route
    M, N, K, kmax = 8, 128, 16384, 4096
    A = fi.uniform((M, K), fi.rng_for(3, 0), 0.0, 1.0, bf16=False)
    B = fi.uniform((N, K), fi.rng_for(3, 1), 0.0, 1.0, bf16=False)
    A8, sA = oracle.quant_1x128(A)
    kb = kmax // 128
    for bmode in (0, 1):
        B8, sB = oracle.quant_128x128(B) if bmode == 0 else oracle.quant_1x128(B)
        ref = oracle.gemm_prefix(A8, sA, B8, sB, kmax, bmode=bmode)
        sBt = sB[:, :kb] if bmode == 0 else sB[:kb]
        cut = oracle.gemm_exact_int(np.ascontiguousarray(A8[:, :kmax]), np.ascontiguousarray(sA[:kb]),
                                    np.ascontiguousarray(B8[:, :kmax]), np.ascontiguousarray(sBt),
                                    bmode=bmode)
        assert np.max(np.abs(ref - cut) / np.abs(cut)) <= 1e-13
        # and the full-K prefix is the full GEMM
        full = oracle.gemm_exact_int(A8, sA, B8, sB, bmode=bmode)
        assert np.max(np.abs(oracle.gemm_prefix(A8, sA, B8, sB, K, bmode=bmode) - full)
                      / np.abs(full)) <= 1e-13
