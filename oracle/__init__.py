"""CPU oracle for the fine-grained FP8 path -- TEST INFRASTRUCTURE ONLY.

Thin numpy/ctypes wrapper over ``fp8q_oracle.c`` (plain C, FP64 GEMM).  Only
``tests/``, the package's ``smoke()`` check and the benchmark's ``cpu_baseline``
leg may import this module.  It imports nothing from the CUDA package and the
CUDA package imports nothing from here.

Each wrapper names the passage it follows; the C source carries the details.
BF16 inputs are passed as numpy ``uint16`` bit patterns and widened exactly to
FP32 here (a BF16 value is the upper half of an FP32 word).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force or an independent library
routine -- except ``gemm_trunc_emu``'s default knobs, which the pages pin only
loosely (one printed figure, ~2% at K=4096, inputs not stated).
"""
import ctypes
import os

import numpy as np

from . import build as _build

GROUP = 128
E4M3_MAX = 448.0

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.fpo_e4m3_decode.restype = ctypes.c_double
        lib.fpo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fpo_e4m3_encode.restype = ctypes.c_uint8
        lib.fpo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fpo_e4m3_decode_array.argtypes = [P, I64, P]
        lib.fpo_e4m3_encode_array.argtypes = [P, I64, P]
        lib.fpo_tile_scale.argtypes = [ctypes.c_float, P, P]
        for name in ("fpo_quant_1x128", "fpo_quant_128x1", "fpo_quant_128x128"):
            getattr(lib, name).argtypes = [P, I64, I64, P, P]
        lib.fpo_retile_1x128_to_128x1.argtypes = [P, P, I64, I64, P, P]
        lib.fpo_swiglu_f64.argtypes = [P, P, I64, P]
        lib.fpo_rmsnorm_f64.argtypes = [P, P, I64, I64, ctypes.c_double, P]
        lib.fpo_gemm_f64.argtypes = [P, P, P, P, I, I64, I64, I64, P, P, I]
        lib.fpo_gemm_f64_entries.argtypes = [P, P, P, P, I, I64, I64, I64, P, P, I64, P, P, I]
        lib.fpo_gemm_grouped_f64.argtypes = [P, P, P, P, P, I64, I64, I64, I64, P, P, I]
        lib.fpo_gemm_grouped_f64_entries.argtypes = [P, P, P, P, P, I64, I64, I64, I64, P, P,
                                                     I64, P, P, I]
        lib.fpo_gemm_exact_int.argtypes = [P, P, P, P, I, I64, I64, I64, P, I]
        lib.fpo_gemm_trunc_emu.argtypes = [P, P, P, P, I, I64, I64, I64, I64, I, I, I, P, I]
        lib.fpo_gemm_f64_prefix.argtypes = [P, P, P, P, I, I64, I64, I64, I64, P, I]
        lib.fpo_max_threads.restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().fpo_max_threads())


def widen(x) -> np.ndarray:
    """FP32 view of an input: float arrays pass through, uint16 is read as BF16 bits."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    return _c(x, np.float32)


# ------------------------------------------------------------------ codec
def e4m3_decode(b) -> np.ndarray:
    """E4M3 byte -> value (FP64), OCP definition; "unified E4M3 format"."""
    b = _c(b, np.uint8)
    out = np.empty(b.shape, np.float64)
    _load().fpo_e4m3_decode_array(_ptr(b), b.size, _ptr(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    """FP32 -> E4M3 byte, round-to-nearest-even, saturating at +-448, NaN -> 0x7F."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().fpo_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def tile_scale(amax: float):
    """(s, inv) for one tile: s = fl32(amax/448), inv = fl32(448/amax)."""
    s = ctypes.c_float()
    inv = ctypes.c_float()
    _load().fpo_tile_scale(ctypes.c_float(amax), ctypes.byref(s), ctypes.byref(inv))
    return np.float32(s.value), np.float32(inv.value)


# ------------------------------------------------------------- quantizers
def _nb(n):
    return (n + GROUP - 1) // GROUP


def quant_1x128(x):
    """Per token per 128 channels ("Six Reasons...", para. 3).  x[M][K] ->
    q[M][K] uint8, s[ceil(K/128)][M] float32."""
    x = widen(x)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((_nb(K), M), np.float32)
    _load().fpo_quant_1x128(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def quant_128x1(x):
    """Per 128 tokens per channel, written transposed ("Six Reasons...", para. 3).
    x[T][C] -> qT[C][T] uint8, sT[ceil(T/128)][C] float32."""
    x = widen(x)
    T, C = x.shape
    q = np.empty((C, T), np.uint8)
    s = np.empty((_nb(T), C), np.float32)
    _load().fpo_quant_128x1(_ptr(x), T, C, _ptr(q), _ptr(s))
    return q, s


def quant_128x128(w):
    """Per 128x128 weight block ("Six Reasons...", para. 3).  w[N][K] ->
    q[N][K] uint8, s[ceil(N/128)][ceil(K/128)] float32."""
    w = widen(w)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((_nb(N), _nb(K)), np.float32)
    _load().fpo_quant_128x128(_ptr(w), N, K, _ptr(q), _ptr(s))
    return q, s


def retile_1x128_to_128x1(q, s):
    """Backward regrouping of stored forward tiles ("Six Reasons...", para. 3):
    dequantize q[T][C] (1x128 scales s[ceil(C/128)][T]) and quantize per 128
    tokens of a channel, transposed: -> qT[C][T], sT[ceil(T/128)][C]."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    T, C = q.shape
    qT = np.empty((C, T), np.uint8)
    sT = np.empty((_nb(T), C), np.float32)
    _load().fpo_retile_1x128_to_128x1(_ptr(q), _ptr(s), T, C, _ptr(qT), _ptr(sT))
    return qT, sT


def swiglu_f64(g, u):
    """SwiGLU(g, u) = silu(g) * u = g u / (1 + e^-g) in FP64 (the SwiGLU
    operator of the woojincopolymer post, para. 4).  g, u: same shape, FP32 or
    BF16 bits."""
    g = widen(g)
    u = widen(u)
    assert g.shape == u.shape
    h = np.empty(g.shape, np.float64)
    _load().fpo_swiglu_f64(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def swiglu_quant_1x128(g, u):
    """Fused SwiGLU + 1x128 FP8 cast (woojincopolymer post, paras. 3-4): the
    exact SwiGLU output rounded once to FP32, quantized per 1x128 tile.
    g, u [M][I] -> (q[M][I] uint8, s[ceil(I/128)][M] float32, h[M][I] FP64)."""
    h = swiglu_f64(g, u)
    q, s = quant_1x128(h.astype(np.float32))
    return q, s, h


def rmsnorm_f64(x, w, eps):
    """RMSNorm y = x w / sqrt(mean(x^2) + eps) per row, in FP64 (the layer
    normalization of the woojincopolymer post, para. 3).  x[M][K], w[K]."""
    x = widen(x)
    w = widen(w)
    M, K = x.shape
    assert w.shape == (K,)
    y = np.empty((M, K), np.float64)
    _load().fpo_rmsnorm_f64(_ptr(x), _ptr(w), M, K, float(eps), _ptr(y))
    return y


def rmsnorm_quant_1x128(x, w, eps):
    """Fused RMSNorm + 1x128 FP8 cast (woojincopolymer post, para. 3): the
    exact normalized value rounded once to FP32, quantized per 1x128 tile.
    -> (q[M][K] uint8, s[ceil(K/128)][M] float32, y[M][K] FP64)."""
    y = rmsnorm_f64(x, w, eps)
    q, s = quant_1x128(y.astype(np.float32))
    return q, s, y


def dequant_1x128(q, s):
    """decode(q) * s per element, in FP64 (exact: both factors are FP32-exact)."""
    q = _c(q, np.uint8)
    M, K = q.shape
    return e4m3_decode(q) * np.repeat(np.asarray(s, np.float64).T, GROUP, axis=1)[:, :K]


# ------------------------------------------------------------------- GEMM
BSCALE_BLOCK128 = 0
BSCALE_ROW1x128 = 1


def gemm(A8, sA, B8, sB, bmode=BSCALE_BLOCK128, threads=0):
    """C = dequant(A8) @ dequant(B8)^T in FP64, plus sum_k |a_k b_k| per entry."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    M, K = A8.shape
    N = B8.shape[0]
    C = np.empty((M, N), np.float64)
    Cabs = np.empty((M, N), np.float64)
    _load().fpo_gemm_f64(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), bmode, M, N, K,
                         _ptr(C), _ptr(Cabs), threads)
    return C, Cabs


def gemm_entries(A8, sA, B8, sB, mi, ni, bmode=BSCALE_BLOCK128, threads=0):
    """The same GEMM evaluated only at entries (mi[i], ni[i])."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    mi, ni = _c(mi, np.int64), _c(ni, np.int64)
    M, K = A8.shape
    N = B8.shape[0]
    C = np.empty(mi.shape, np.float64)
    Cabs = np.empty(mi.shape, np.float64)
    _load().fpo_gemm_f64_entries(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), bmode, M, N, K,
                                 _ptr(mi), _ptr(ni), mi.size, _ptr(C), _ptr(Cabs), threads)
    return C, Cabs


def gemm_grouped(A8, sA, B8, sB, m_offsets, threads=0):
    """MoE grouped GEMM ([P4] item 8): group e's rows times its own B8[e]."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    mo = _c(m_offsets, np.int64)
    Mtot, K = A8.shape
    G, N, _ = B8.shape
    C = np.zeros((Mtot, N), np.float64)
    Cabs = np.zeros((Mtot, N), np.float64)
    _load().fpo_gemm_grouped_f64(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), _ptr(mo), G, Mtot, N,
                                 K, _ptr(C), _ptr(Cabs), threads)
    return C, Cabs


def gemm_grouped_entries(A8, sA, B8, sB, m_offsets, mi, ni, threads=0):
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    mo = _c(m_offsets, np.int64)
    mi, ni = _c(mi, np.int64), _c(ni, np.int64)
    Mtot, K = A8.shape
    G, N, _ = B8.shape
    C = np.empty(mi.shape, np.float64)
    Cabs = np.empty(mi.shape, np.float64)
    _load().fpo_gemm_grouped_f64_entries(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), _ptr(mo), G,
                                         Mtot, N, K, _ptr(mi), _ptr(ni), mi.size, _ptr(C),
                                         _ptr(Cabs), threads)
    return C, Cabs


def gemm_exact_int(A8, sA, B8, sB, bmode=BSCALE_BLOCK128, threads=0):
    """Independent route: exact int64 group sums, then FP64 scaling."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    M, K = A8.shape
    N = B8.shape[0]
    C = np.empty((M, N), np.float64)
    _load().fpo_gemm_exact_int(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), bmode, M, N, K,
                               _ptr(C), threads)
    return C


def gemm_trunc_emu(A8, sA, B8, sB, kmax=None, chunk=4, mbits=13, promote=0,
                   bmode=BSCALE_BLOCK128, threads=0):
    """Limited-precision accumulation stand-in ("Six Reasons...", paras. 2-3).

    promote=0: no promotion over the first kmax elements of K.
    promote=P: the limited accumulator restarts every P elements and partials
    are summed in FP64 (promotion)."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    M, K = A8.shape
    N = B8.shape[0]
    kmax = K if kmax is None else int(kmax)
    C = np.empty((M, N), np.float64)
    _load().fpo_gemm_trunc_emu(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), bmode, M, N, K, kmax,
                               chunk, mbits, promote, _ptr(C), threads)
    return C


def gemm_prefix(A8, sA, B8, sB, kmax, bmode=BSCALE_BLOCK128, threads=0):
    """FP64 GEMM over the first kmax elements of K (for the emulator's error)."""
    A8, B8 = _c(A8, np.uint8), _c(B8, np.uint8)
    sA, sB = _c(sA, np.float32), _c(sB, np.float32)
    M, K = A8.shape
    N = B8.shape[0]
    C = np.empty((M, N), np.float64)
    _load().fpo_gemm_f64_prefix(_ptr(A8), _ptr(sA), _ptr(B8), _ptr(sB), bmode, M, N, K,
                                int(kmax), _ptr(C), threads)
    return C


# ------------------------------------------------------ expert-parallel MoE
def bf16_round(x):
    """FP64 -> nearest BF16 value (as FP64), ties to even: the rounding of a
    BF16 output.  Plain definition: x = m 2^e with 1/2 <= |m| < 1 (frexp,
    exact); BF16 keeps 8 significant bits, so the result is rint(256 m) 2^(e-8)
    with numpy's rint rounding halves to even (a carry to 256 lands on the
    next power of two, which is representable).  Finite, normal-range values."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def moe_ep_reference(x, topk_ids, topk_w, W8, sW):
    """Expert-parallel MoE layer with FP8 dispatch and BF16 combine ("Six
    Reasons Deepseek Ai Is A Waste Of Time", para. 4: the activations are
    quantized to FP8 before they are dispatched to the experts' up
    projection, and the combine stays in BF16).  Token t's activations are
    quantized per 1x128 tile; for each of its k experts e = topk_ids[t][j] the
    expert's block-scaled FP8 GEMM gives y_tj = dequant(q_t) . dequant(W8_e)^T
    (FP64 here), returned as BF16; the output is
        out[t] = bf16( sum_j topk_w[t][j] * bf16(y_tj) ).
      x        [T][H] activations (BF16 bits as uint16, or FP32)
      topk_ids [T][k] expert ids in [0, E), distinct within a row
      topk_w   [T][k] gate weights (FP32)
      W8, sW   [E][N][H] uint8, [E][N/128][H/128] float32: the experts'
               weights quantized per 128x128 block
    Returns (out [T][N], y [T][k][N] exact expert results, yabs [T][k][N]
    sum_h |a_h b_h|), all FP64; out holds BF16 values."""
    q, s = quant_1x128(x)
    ids = np.asarray(topk_ids, np.int64)
    w = np.asarray(topk_w, np.float32).astype(np.float64)
    T, k = ids.shape
    E, N, H = W8.shape
    y = np.zeros((T, k, N))
    yabs = np.zeros((T, k, N))
    for e in range(E):
        ts, js = np.nonzero(ids == e)
        if ts.size == 0:
            continue
        Ce, Ca = gemm(q[ts], s[:, ts], W8[e], sW[e])
        y[ts, js] = Ce
        yabs[ts, js] = Ca
    out = bf16_round(np.einsum("tk,tkn->tn", w, bf16_round(y)))
    return out, y, yabs
