"""Pins of the oracle's block-scaled GEMM (CPU only).

Against: numpy matmul on operands decoded by torch's float8_e4m3fn (an
independent decoder and an independent summation), exact rational brute force
on tiny shapes, the oracle's own exact-int64 route, and closed forms
(constant operands, one-hot selection).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import fp8q_inputs as fi


def torch_decode(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_rows(q8, s_kb_rows):
    """q8[R][K] with scales s[Kb][R] -> FP64 [R][K]."""
    R, K = q8.shape
    sfull = np.repeat(s_kb_rows.T.astype(np.float64), 128, axis=1)[:, :K]
    return torch_decode(q8) * sfull


def dequant_blocks(q8, s_nb_kb):
    N, K = q8.shape
    sfull = np.repeat(np.repeat(s_nb_kb.astype(np.float64), 128, axis=0), 128, axis=1)[:N, :K]
    return torch_decode(q8) * sfull


def make_operands(oracle, M, N, K, seed, bmode=0):
    A = fi.gaussian((M, K), fi.rng_for(seed, 0), 1.0, 0.01, 100.0, bf16=False)
    B = fi.gaussian((N, K), fi.rng_for(seed, 1), 0.02, bf16=False)
    A8, sA = oracle.quant_1x128(A)
    if bmode == 0:
        B8, sB = oracle.quant_128x128(B)
    else:
        B8, sB = oracle.quant_1x128(B)
    return A8, sA, B8, sB


@pytest.mark.parametrize("M,N,K", [(128, 128, 512), (70, 200, 384), (33, 129, 200)])
def test_gemm_matches_numpy_block128(oracle, M, N, K):
    A8, sA, B8, sB = make_operands(oracle, M, N, K, seed=M + N + K)
    C, Cabs = oracle.gemm(A8, sA, B8, sB)
    ref = dequant_rows(A8, sA) @ dequant_blocks(B8, sB).T
    refabs = np.abs(dequant_rows(A8, sA)) @ np.abs(dequant_blocks(B8, sB)).T
    assert np.all(np.abs(C - ref) <= 1e-12 * refabs + 1e-300)
    assert np.allclose(Cabs, refabs, rtol=1e-12, atol=0)


def test_gemm_matches_numpy_row_scales(oracle):
    M, N, K = 96, 160, 384
    A8, sA, B8, sB = make_operands(oracle, M, N, K, seed=5, bmode=1)
    C, _ = oracle.gemm(A8, sA, B8, sB, bmode=oracle.BSCALE_ROW1x128)
    ref = dequant_rows(A8, sA) @ dequant_rows(B8, sB).T
    refabs = np.abs(dequant_rows(A8, sA)) @ np.abs(dequant_rows(B8, sB)).T
    assert np.all(np.abs(C - ref) <= 1e-12 * refabs)


@pytest.mark.parametrize("bmode", [0, 1])
def test_exact_integer_route_agrees(oracle, bmode):
    A8, sA, B8, sB = make_operands(oracle, 64, 256, 640, seed=9, bmode=bmode)
    C, Cabs = oracle.gemm(A8, sA, B8, sB, bmode=bmode)
    Cx = oracle.gemm_exact_int(A8, sA, B8, sB, bmode=bmode)
    assert np.all(np.abs(C - Cx) <= 1e-13 * Cabs)


def test_brute_force_exact_rationals(oracle):
    """Tiny shapes summed exactly with Python Fractions, random byte patterns."""
    rng = np.random.default_rng(3)
    finite = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], np.uint8)
    dec = {int(b): Fraction(float(v)) for b, v in zip(finite, torch_decode(finite))}
    for M, N, K in [(1, 1, 128), (3, 4, 128), (4, 2, 256), (2, 3, 200)]:
        Kb = (K + 127) // 128
        Nb = (N + 127) // 128
        A8 = rng.choice(finite, size=(M, K))
        B8 = rng.choice(finite, size=(N, K))
        sA = rng.uniform(1e-3, 4, size=(Kb, M)).astype(np.float32)
        sB = rng.uniform(1e-3, 4, size=(Nb, Kb)).astype(np.float32)
        C, _ = oracle.gemm(A8, sA, B8, sB)
        for m in range(M):
            for n in range(N):
                exact = sum(dec[int(A8[m, k])] * Fraction(float(sA[k // 128, m]))
                            * dec[int(B8[n, k])] * Fraction(float(sB[n // 128, k // 128]))
                            for k in range(K))
                assert abs(Fraction(C[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 45) + \
                    Fraction(1, 2 ** 200)


def test_constant_operands_closed_form(oracle):
    M, N, K = 8, 8, 512
    a_code, b_code = 0x44, 0xB9          # 3.0 and -1.125
    A8 = np.full((M, K), a_code, np.uint8)
    B8 = np.full((N, K), b_code, np.uint8)
    sA = np.full((K // 128, M), 0.5, np.float32)
    sB = np.full((1, K // 128), 2.0, np.float32)
    C, Cabs = oracle.gemm(A8, sA, B8, sB)
    assert np.all(C == K * 3.0 * 0.5 * (-1.125) * 2.0)
    assert np.all(Cabs == -C)


def test_one_hot_selects_columns(oracle):
    M, N, K = 16, 128, 256
    perm = np.random.default_rng(4).permutation(K)[:M]
    A8 = np.zeros((M, K), np.uint8)
    A8[np.arange(M), perm] = 0x38          # 1.0
    sA = np.ones((K // 128, M), np.float32)
    B = fi.gaussian((N, K), fi.rng_for(21, 0), bf16=False)
    B8, sB = oracle.quant_128x128(B)
    C, _ = oracle.gemm(A8, sA, B8, sB)
    Bd = dequant_blocks(B8, sB)
    assert np.array_equal(C, Bd[:, perm].T)


def test_entries_match_full(oracle):
    A8, sA, B8, sB = make_operands(oracle, 64, 128, 384, seed=31)
    C, Cabs = oracle.gemm(A8, sA, B8, sB)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, 64, 100)
    ni = rng.integers(0, 128, 100)
    Ce, Cae = oracle.gemm_entries(A8, sA, B8, sB, mi, ni)
    assert np.array_equal(Ce, C[mi, ni]) and np.array_equal(Cae, Cabs[mi, ni])


def test_grouped_matches_per_group_numpy(oracle):
    sizes = np.array([128, 0, 256, 128], np.int64)
    offs = fi.offsets_from_sizes(sizes)
    Mtot, G, N, K = int(offs[-1]), len(sizes), 128, 384
    A = fi.gaussian((Mtot, K), fi.rng_for(41, 0), 1.0, 0.01, 100.0, bf16=False)
    W = fi.gaussian((G, N, K), fi.rng_for(41, 1), 0.02, bf16=False)
    A8, sA = oracle.quant_1x128(A)
    B8 = np.empty((G, N, K), np.uint8)
    sB = np.empty((G, 1, 3), np.float32)
    for e in range(G):
        B8[e], sB[e] = oracle.quant_128x128(W[e])
    C, _ = oracle.gemm_grouped(A8, sA, B8, sB, offs)
    Ad = dequant_rows(A8, sA)
    for e in range(G):
        r0, r1 = offs[e], offs[e + 1]
        ref = Ad[r0:r1] @ dequant_blocks(B8[e], sB[e]).T
        absref = np.abs(Ad[r0:r1]) @ np.abs(dequant_blocks(B8[e], sB[e])).T
        assert np.all(np.abs(C[r0:r1] - ref) <= 1e-12 * absref)
    mi = np.array([0, 127, 128, 300, 511])
    ni = np.array([0, 5, 127, 64, 100])
    Ce, _ = oracle.gemm_grouped_entries(A8, sA, B8, sB, offs, mi, ni)
    assert np.array_equal(Ce, C[mi, ni])
