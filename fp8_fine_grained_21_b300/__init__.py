"""fp8q: fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM on B300.

Thin ctypes binding over ``libfp8q.so`` (C ABI in ``include/fp8q.h``).  The
functions named ``fp8q_*`` mirror the C entry points one to one and take torch
CUDA tensors for every buffer; the short-named helpers allocate the outputs
with torch and call them.  Torch supplies device memory and streams only:
every step of the computation runs in the library's CUDA kernels.  There is no
CPU fallback -- if the library is missing or a tensor is not on a CUDA device,
the call raises.
"""
import ctypes
import os

import torch

__all__ = [
    "Fp8qError", "library_path", "load",
    "fp8q_quant_act_1x128", "fp8q_quant_act_128x1", "fp8q_quant_w_128x128",
    "fp8q_retile_1x128_to_128x1", "fp8q_transpose_w_128x128", "retile_1x128_to_128x1",
    "transpose_w_128x128",
    "fp8q_gemm", "fp8q_gemm_ex", "fp8q_gemm_grouped", "fp8q_gemm_ws", "fp8q_gemm_grouped_ws",
    "fp8q_gemm_workspace_size", "fp8q_gemm_noalloc", "fp8q_gemm_quant_a", "gemm_quant_a",
    "fp8q_ep_row_bytes", "fp8q_ep_route", "fp8q_ep_pack", "fp8q_ep_unpack", "fp8q_ep_gather",
    "fp8q_ep_combine", "fp8q_get_device_status",
    "fp8q_selftest_wait", "fp8q_bench_mma_peak", "fp8q_num_sms", "fp8q_status_string",
    "fp8q_version", "workspace",
    "quant_act_1x128", "quant_act_128x1", "quant_w_128x128", "gemm", "gemm_grouped",
    "F32", "BF16", "BSCALE_BLOCK128", "BSCALE_ROW1x128",
]

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libfp8q.so")

F32, BF16 = 0, 1
BSCALE_BLOCK128, BSCALE_ROW1x128 = 0, 1
STATUS_NAMES = {0: "FP8Q_OK", 1: "FP8Q_ERR_INVALID_ARG", 2: "FP8Q_ERR_UNSUPPORTED_SHAPE",
                3: "FP8Q_ERR_MISALIGNED", 4: "FP8Q_ERR_CUDA", 5: "FP8Q_ERR_TIMEOUT",
                6: "FP8Q_ERR_BAD_GROUPS", 7: "FP8Q_ERR_BAD_ROUTING"}
EXPORTS = ("fp8q_quant_act_1x128", "fp8q_quant_act_128x1", "fp8q_quant_w_128x128",
           "fp8q_swiglu_quant_1x128", "fp8q_rmsnorm_quant_1x128",
           "fp8q_retile_1x128_to_128x1", "fp8q_transpose_w_128x128", "fp8q_gemm",
           "fp8q_gemm_ex", "fp8q_gemm_grouped", "fp8q_gemm_ws", "fp8q_gemm_grouped_ws",
           "fp8q_gemm_workspace_size", "fp8q_gemm_noalloc", "fp8q_gemm_quant_a",
           "fp8q_ep_row_bytes", "fp8q_ep_route", "fp8q_ep_pack", "fp8q_ep_unpack",
           "fp8q_ep_gather", "fp8q_ep_combine", "fp8q_get_device_status",
           "fp8q_selftest_wait", "fp8q_bench_mma_peak", "fp8q_num_sms", "fp8q_status_string",
           "fp8q_version")


class Fp8qError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, STATUS_NAMES.get(status, "?"), status))


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libfp8q.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("fp8q CUDA library not built (%s missing); run "
                           "`python -m fp8_fine_grained_21_b300.build`" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    for name in ("fp8q_quant_act_1x128", "fp8q_quant_act_128x1", "fp8q_quant_w_128x128"):
        f = getattr(lib, name)
        f.argtypes = [P, I, I64, I64, P, P, P]
        f.restype = I
    lib.fp8q_swiglu_quant_1x128.argtypes = [P, P, I, I64, I64, I64, P, P, P]
    lib.fp8q_swiglu_quant_1x128.restype = I
    lib.fp8q_rmsnorm_quant_1x128.argtypes = [P, P, I, I64, I64, ctypes.c_float, P, P, P]
    lib.fp8q_rmsnorm_quant_1x128.restype = I
    for name in ("fp8q_retile_1x128_to_128x1", "fp8q_transpose_w_128x128"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I64, I64, P, P, P]
        f.restype = I
    lib.fp8q_gemm.argtypes = [P, P, P, P, P, I64, I64, I64, I]
    lib.fp8q_gemm.restype = I
    lib.fp8q_gemm_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P]
    lib.fp8q_gemm_ex.restype = I
    lib.fp8q_gemm_grouped.argtypes = [P, P, P, P, P, P, I, I64, I64, I64, I, P]
    lib.fp8q_gemm_grouped.restype = I
    SZ = ctypes.c_size_t
    lib.fp8q_gemm_ws.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P]
    lib.fp8q_gemm_ws.restype = I
    lib.fp8q_gemm_grouped_ws.argtypes = [P, P, P, P, P, P, I, I64, I64, I64, I, P, SZ, P]
    lib.fp8q_gemm_grouped_ws.restype = I
    lib.fp8q_gemm_workspace_size.argtypes = []
    lib.fp8q_gemm_workspace_size.restype = SZ
    lib.fp8q_gemm_noalloc.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P]
    lib.fp8q_gemm_noalloc.restype = I
    lib.fp8q_gemm_quant_a.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, P, SZ, P]
    lib.fp8q_gemm_quant_a.restype = I
    lib.fp8q_ep_row_bytes.argtypes = [I64]
    lib.fp8q_ep_row_bytes.restype = I64
    lib.fp8q_ep_route.argtypes = [P, I64, I, I, P, P, P]
    lib.fp8q_ep_route.restype = I
    lib.fp8q_ep_pack.argtypes = [P, P, P, I64, I, I64, P, P]
    lib.fp8q_ep_pack.restype = I
    lib.fp8q_ep_unpack.argtypes = [P, I64, I64, P, P, I, P, P, I, P, P, I64, P]
    lib.fp8q_ep_unpack.restype = I
    lib.fp8q_ep_gather.argtypes = [P, I64, I64, I64, P, P, I, P, P]
    lib.fp8q_ep_gather.restype = I
    lib.fp8q_ep_combine.argtypes = [P, P, P, I64, I, I64, P, P]
    lib.fp8q_ep_combine.restype = I
    lib.fp8q_selftest_wait.argtypes = [I64, P]
    lib.fp8q_selftest_wait.restype = I
    lib.fp8q_bench_mma_peak.argtypes = [I64, P]
    lib.fp8q_bench_mma_peak.restype = I
    lib.fp8q_num_sms.argtypes = []
    lib.fp8q_num_sms.restype = I
    lib.fp8q_get_device_status.argtypes = [P]
    lib.fp8q_get_device_status.restype = I
    lib.fp8q_status_string.argtypes = [I]
    lib.fp8q_status_string.restype = ctypes.c_char_p
    lib.fp8q_version.argtypes = []
    lib.fp8q_version.restype = I
    _lib = lib
    return lib


# ---------------------------------------------------------------- marshalling
_IN_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}


def _dev(t: torch.Tensor, name: str, dtype=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, rc):
    if rc != 0:
        raise Fp8qError(fn, rc)


def _in_dtype(x):
    try:
        return _IN_DTYPES[x.dtype]
    except KeyError:
        raise ValueError("input must be float32 or bfloat16, got %s" % x.dtype) from None


def _out_dtype(dt):
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError("output must be float32 or bfloat16, got %s" % dt)


def _shape(t, name, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _numel(t, name, n):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.numel() != n:
        raise ValueError("%s must hold %d elements, got %d" % (name, n, t.numel()))


def _gemm_dims(A8, B8, C, sA, sB, bscale, grouped=False):
    """(M, N, K[, G]) of a GEMM call, after checking that every buffer has the
    size the library will read or write: A8 [M][K]; B8 [N][K] ([G][N][K]
    grouped); C [M][N]; sA [K/128][M]; sB [N/128][K/128] ([G][..] grouped) for
    128x128 blocks or [K/128][N] for 1x128 rows.  The library trusts these
    sizes, so a mismatch here would otherwise read or write out of bounds."""
    if A8.dim() != 2:
        raise ValueError("A8 must be 2-D [M][K]")
    M, K = A8.shape
    if grouped:
        if B8.dim() != 3:
            raise ValueError("B8 must be 3-D [G][N][K]")
        G, N, Kb_ = B8.shape
    else:
        if B8.dim() != 2:
            raise ValueError("B8 must be 2-D [N][K]")
        G = 1
        N, Kb_ = B8.shape
    if Kb_ != K:
        raise ValueError("A8 and B8 must have the same K (%d vs %d)" % (K, Kb_))
    _shape(C, "C", (M, N))
    kb, nb = _scales(K), _scales(N)
    _numel(sA, "sA", kb * M)
    if bscale == BSCALE_ROW1x128:
        _numel(sB, "sB", kb * N)
    elif bscale == BSCALE_BLOCK128:
        _numel(sB, "sB", G * nb * kb)
    else:
        raise ValueError("bscale must be BSCALE_BLOCK128 or BSCALE_ROW1x128")
    return (M, N, K, G) if grouped else (M, N, K)


def _quant_out(q, s, q_shape, s_numel):
    _shape(q, "q", q_shape)
    _numel(s, "s", s_numel)


# ------------------------------------------------------- same-name bindings
def fp8q_quant_act_1x128(x, q, s, stream=None):
    M, K = x.shape
    _quant_out(q, s, (M, K), _scales(K) * M)
    _check("fp8q_quant_act_1x128", load().fp8q_quant_act_1x128(
        _dev(x, "x"), _in_dtype(x), M, K, _dev(q, "q", torch.uint8),
        _dev(s, "s", torch.float32), _stream(stream)))


def _rows(t: torch.Tensor, name: str):
    """Pointer and row stride (elements) of a 2-D CUDA tensor with unit column stride."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (no CPU path)" % name)
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be 2-D with unit column stride" % name)
    return ctypes.c_void_p(t.data_ptr()), t.stride(0)


def fp8q_swiglu_quant_1x128(gate, up, q, s, stream=None):
    """gate, up: [M][I] views with the same row stride (e.g. the two halves of
    a [M][2I] projection output)."""
    if gate.shape != up.shape or gate.dtype != up.dtype:
        raise ValueError("gate and up must have the same shape and dtype")
    pg, ld = _rows(gate, "gate")
    pu, ldu = _rows(up, "up")
    if ldu != ld:
        raise ValueError("gate and up must have the same row stride")
    M, I = gate.shape
    _quant_out(q, s, (M, I), _scales(I) * M)
    _check("fp8q_swiglu_quant_1x128", load().fp8q_swiglu_quant_1x128(
        pg, pu, _in_dtype(gate), M, I, ld, _dev(q, "q", torch.uint8),
        _dev(s, "s", torch.float32), _stream(stream)))


def fp8q_rmsnorm_quant_1x128(x, w, q, s, eps=1e-6, stream=None):
    """x [M][K], w [K] (same dtype); eps > 0."""
    M, K = x.shape
    if w.dtype != x.dtype or tuple(w.shape) != (K,):
        raise ValueError("w must be [K] with x's dtype")
    _quant_out(q, s, (M, K), _scales(K) * M)
    _check("fp8q_rmsnorm_quant_1x128", load().fp8q_rmsnorm_quant_1x128(
        _dev(x, "x"), _dev(w, "w"), _in_dtype(x), M, K, ctypes.c_float(eps),
        _dev(q, "q", torch.uint8), _dev(s, "s", torch.float32), _stream(stream)))


def fp8q_quant_act_128x1(x, qT, sT, stream=None):
    T, C = x.shape
    _shape(qT, "qT", (C, T))
    _numel(sT, "sT", _scales(T) * C)
    _check("fp8q_quant_act_128x1", load().fp8q_quant_act_128x1(
        _dev(x, "x"), _in_dtype(x), T, C, _dev(qT, "qT", torch.uint8),
        _dev(sT, "sT", torch.float32), _stream(stream)))


def fp8q_quant_w_128x128(w, q, s, stream=None):
    N, K = w.shape
    _quant_out(q, s, (N, K), _scales(N) * _scales(K))
    _check("fp8q_quant_w_128x128", load().fp8q_quant_w_128x128(
        _dev(w, "w"), _in_dtype(w), N, K, _dev(q, "q", torch.uint8),
        _dev(s, "s", torch.float32), _stream(stream)))


def fp8q_retile_1x128_to_128x1(q, s, qT, sT, stream=None):
    T, C = q.shape
    _numel(s, "s", _scales(C) * T)
    _shape(qT, "qT", (C, T))
    _numel(sT, "sT", _scales(T) * C)
    _check("fp8q_retile_1x128_to_128x1", load().fp8q_retile_1x128_to_128x1(
        _dev(q, "q", torch.uint8), _dev(s, "s", torch.float32), T, C, _dev(qT, "qT", torch.uint8),
        _dev(sT, "sT", torch.float32), _stream(stream)))


def fp8q_transpose_w_128x128(q, s, qT, sT, stream=None):
    N, K = q.shape
    _numel(s, "s", _scales(N) * _scales(K))
    _shape(qT, "qT", (K, N))
    _numel(sT, "sT", _scales(K) * _scales(N))
    _check("fp8q_transpose_w_128x128", load().fp8q_transpose_w_128x128(
        _dev(q, "q", torch.uint8), _dev(s, "s", torch.float32), N, K, _dev(qT, "qT", torch.uint8),
        _dev(sT, "sT", torch.float32), _stream(stream)))


def fp8q_gemm(A8, sA, B8, sB, C):
    M, N, K = _gemm_dims(A8, B8, C, sA, sB, BSCALE_BLOCK128)
    _check("fp8q_gemm", load().fp8q_gemm(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), M, N, K, _out_dtype(C.dtype)))


def fp8q_gemm_ex(A8, sA, B8, sB, C, bscale=BSCALE_BLOCK128, stream=None):
    M, N, K = _gemm_dims(A8, B8, C, sA, sB, bscale)
    _check("fp8q_gemm_ex", load().fp8q_gemm_ex(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), M, N, K, _out_dtype(C.dtype), int(bscale),
        _stream(stream)))


def fp8q_gemm_grouped(A8, sA, B8, sB, C, m_offsets, stream=None):
    Mtot, N, K, G = _gemm_dims(A8, B8, C, sA, sB, BSCALE_BLOCK128, grouped=True)
    _numel(m_offsets, "m_offsets", G + 1)
    _check("fp8q_gemm_grouped", load().fp8q_gemm_grouped(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), _dev(m_offsets, "m_offsets", torch.int32),
        G, Mtot, N, K, _out_dtype(C.dtype), _stream(stream)))


def _ws(ws):
    if ws is None:
        return ctypes.c_void_p(None), 0
    return _dev(ws, "workspace", torch.uint8), ws.numel()


def fp8q_gemm_ws(A8, sA, B8, sB, C, bscale=BSCALE_BLOCK128, ws=None, stream=None):
    M, N, K = _gemm_dims(A8, B8, C, sA, sB, bscale)
    wp, wn = _ws(ws)
    _check("fp8q_gemm_ws", load().fp8q_gemm_ws(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), M, N, K, _out_dtype(C.dtype), int(bscale),
        wp, wn, _stream(stream)))


def fp8q_gemm_grouped_ws(A8, sA, B8, sB, C, m_offsets, ws=None, stream=None):
    Mtot, N, K, G = _gemm_dims(A8, B8, C, sA, sB, BSCALE_BLOCK128, grouped=True)
    _numel(m_offsets, "m_offsets", G + 1)
    wp, wn = _ws(ws)
    _check("fp8q_gemm_grouped_ws", load().fp8q_gemm_grouped_ws(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), _dev(m_offsets, "m_offsets", torch.int32),
        G, Mtot, N, K, _out_dtype(C.dtype), wp, wn, _stream(stream)))


def fp8q_gemm_noalloc(A8, sA, B8, sB, C, bscale=BSCALE_BLOCK128, stream=None):
    """The stream-K GEMM on the library's own scratch array (no allocation)."""
    M, N, K = _gemm_dims(A8, B8, C, sA, sB, bscale)
    _check("fp8q_gemm_noalloc", load().fp8q_gemm_noalloc(
        _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32), _dev(B8, "B8", torch.uint8),
        _dev(sB, "sB", torch.float32), _dev(C, "C"), M, N, K, _out_dtype(C.dtype), int(bscale),
        _stream(stream)))


def fp8q_gemm_quant_a(A, B8, sB, C, A8_out=None, sA_out=None, ws=None, stream=None):
    """GEMM on BF16 activations quantized 1x128 inside the kernel; optionally
    also writes the quantized activations (A8_out [M][K] uint8, sA_out
    [K/128][M] float32, both or neither)."""
    if A.dim() != 2 or B8.dim() != 2:
        raise ValueError("A must be [M][K] and B8 [N][K]")
    M, K = A.shape
    N, Kb_ = B8.shape
    if Kb_ != K:
        raise ValueError("A and B8 must have the same K (%d vs %d)" % (K, Kb_))
    _shape(C, "C", (M, N))
    _numel(sB, "sB", _scales(N) * _scales(K))
    if (A8_out is None) != (sA_out is None):
        raise ValueError("give both A8_out and sA_out, or neither")
    if A8_out is not None:
        _shape(A8_out, "A8_out", (M, K))
        _numel(sA_out, "sA_out", _scales(K) * M)
        pa, ps = _dev(A8_out, "A8_out", torch.uint8), _dev(sA_out, "sA_out", torch.float32)
    else:
        pa, ps = ctypes.c_void_p(None), ctypes.c_void_p(None)
    wp, wn = _ws(ws)
    _check("fp8q_gemm_quant_a", load().fp8q_gemm_quant_a(
        _dev(A, "A", torch.bfloat16), _dev(B8, "B8", torch.uint8), _dev(sB, "sB", torch.float32),
        _dev(C, "C"), pa, ps, M, N, K, _out_dtype(C.dtype), wp, wn, _stream(stream)))


# ------------------------------------------- expert-parallel MoE data path
def _opt(t, name, dtype=None):
    """Device pointer of t, or NULL for an empty tensor (a rank may send or
    receive no rows)."""
    if t.numel() == 0:
        return ctypes.c_void_p(None)
    return _dev(t, name, dtype)


def fp8q_ep_row_bytes(H: int) -> int:
    n = int(load().fp8q_ep_row_bytes(int(H)))
    if n < 0:
        raise ValueError("H must be a positive multiple of 128")
    return n


def fp8q_ep_route(topk_ids, E, counts, pos, stream=None):
    if topk_ids.dim() != 2:
        raise ValueError("topk_ids must be [T][k]")
    T, k = topk_ids.shape
    _numel(counts, "counts", E)
    _shape(pos, "pos", (T, k))
    _check("fp8q_ep_route", load().fp8q_ep_route(
        _dev(topk_ids, "topk_ids", torch.int32), T, k, int(E), _dev(counts, "counts", torch.int32),
        _dev(pos, "pos", torch.int32), _stream(stream)))


def fp8q_ep_pack(q, s, pos, send, stream=None):
    T, H = q.shape
    k = pos.shape[1] if pos.dim() == 2 else 1
    _numel(s, "s", _scales(H) * T)
    _shape(pos, "pos", (T, k))
    _shape(send, "send", (T * k, fp8q_ep_row_bytes(H)))
    _check("fp8q_ep_pack", load().fp8q_ep_pack(
        _opt(q, "q", torch.uint8), _opt(s, "s", torch.float32), _opt(pos, "pos", torch.int32),
        T, k, H, _opt(send, "send", torch.uint8), _stream(stream)))


def fp8q_ep_unpack(recv, src_off, dest_base, m_offsets, rows_e, A8, sA, stream=None):
    Mp, H = A8.shape
    R = recv.shape[0]
    nb = dest_base.numel()
    El = rows_e.numel()
    _shape(recv, "recv", (R, fp8q_ep_row_bytes(H)))
    _numel(src_off, "src_off", nb + 1)
    _numel(m_offsets, "m_offsets", El + 1)
    _numel(sA, "sA", _scales(H) * Mp)
    i64 = torch.int64
    _check("fp8q_ep_unpack", load().fp8q_ep_unpack(
        _opt(recv, "recv", torch.uint8), R, H, _dev(src_off, "src_off", i64),
        _dev(dest_base, "dest_base", i64), nb, _dev(m_offsets, "m_offsets", i64),
        _dev(rows_e, "rows_e", i64), El, _dev(A8, "A8", torch.uint8), _dev(sA, "sA", torch.float32),
        Mp, _stream(stream)))


def fp8q_ep_gather(Y, src_off, dest_base, out, stream=None):
    Mp, N = Y.shape
    R = out.shape[0]
    nb = dest_base.numel()
    _shape(out, "out", (R, N))
    _numel(src_off, "src_off", nb + 1)
    i64 = torch.int64
    _check("fp8q_ep_gather", load().fp8q_ep_gather(
        _dev(Y, "Y", torch.bfloat16), Mp, R, N, _dev(src_off, "src_off", i64),
        _dev(dest_base, "dest_base", i64), nb, _opt(out, "out", torch.bfloat16), _stream(stream)))


def fp8q_ep_combine(back, pos, w, out, stream=None):
    T, k = pos.shape
    N = out.shape[1]
    _shape(back, "back", (T * k, N))
    _shape(w, "w", (T, k))
    _shape(out, "out", (T, N))
    _check("fp8q_ep_combine", load().fp8q_ep_combine(
        _opt(back, "back", torch.bfloat16), _opt(pos, "pos", torch.int32),
        _opt(w, "w", torch.float32), T, k, N, _opt(out, "out", torch.bfloat16), _stream(stream)))


def fp8q_gemm_workspace_size() -> int:
    return int(load().fp8q_gemm_workspace_size())


_WORKSPACES = {}


def workspace(device=None, stream=None):
    """Zero-initialised stream-K workspace for (device, stream), allocated with
    torch on first use and kept; calls leave its counters zero again."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    key = (dev.index, int(stream.cuda_stream) if isinstance(stream, torch.cuda.Stream) else int(stream))
    ws = _WORKSPACES.get(key)
    if ws is None:
        with torch.cuda.device(dev):
            n = fp8q_gemm_workspace_size()
            if n == 0:
                raise Fp8qError("fp8q_gemm_workspace_size", 4)
            ws = torch.zeros(n, dtype=torch.uint8, device=dev)
        _WORKSPACES[key] = ws
    return ws


def fp8q_get_device_status(stream=None) -> int:
    return int(load().fp8q_get_device_status(_stream(stream)))


def fp8q_selftest_wait(limit_ns: int, stream=None):
    _check("fp8q_selftest_wait", load().fp8q_selftest_wait(int(limit_ns), _stream(stream)))


def fp8q_bench_mma_peak(blocks: int, stream=None):
    _check("fp8q_bench_mma_peak", load().fp8q_bench_mma_peak(int(blocks), _stream(stream)))


def fp8q_num_sms() -> int:
    n = int(load().fp8q_num_sms())
    if n <= 0:
        raise Fp8qError("fp8q_num_sms", -n)
    return n


def fp8q_status_string(status: int) -> str:
    return load().fp8q_status_string(int(status)).decode()


def fp8q_version() -> int:
    return int(load().fp8q_version())


# -------------------------------------------------------- allocating helpers
def _scales(n):
    return (n + 127) // 128


def quant_act_1x128(x, stream=None):
    """x[M][K] -> (q[M][K] uint8 E4M3, s[K/128][M] float32)."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((_scales(K), M), dtype=torch.float32, device=x.device)
    fp8q_quant_act_1x128(x, q, s, stream)
    return q, s


def swiglu_quant_1x128(gate, up, stream=None):
    """silu(gate) * up, quantized 1x128: -> (q[M][I] uint8, s[I/128][M] float32)."""
    M, I = gate.shape
    q = torch.empty((M, I), dtype=torch.uint8, device=gate.device)
    s = torch.empty((_scales(I), M), dtype=torch.float32, device=gate.device)
    fp8q_swiglu_quant_1x128(gate, up, q, s, stream)
    return q, s


def rmsnorm_quant_1x128(x, w, eps=1e-6, stream=None):
    """RMSNorm(x) * w, quantized 1x128: -> (q[M][K] uint8, s[K/128][M] float32)."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((_scales(K), M), dtype=torch.float32, device=x.device)
    fp8q_rmsnorm_quant_1x128(x, w, q, s, eps, stream)
    return q, s


def quant_act_128x1(x, stream=None):
    """x[T][C] -> (qT[C][T] uint8, sT[T/128][C] float32)."""
    T, C = x.shape
    q = torch.empty((C, T), dtype=torch.uint8, device=x.device)
    s = torch.empty((_scales(T), C), dtype=torch.float32, device=x.device)
    fp8q_quant_act_128x1(x, q, s, stream)
    return q, s


def quant_w_128x128(w, stream=None):
    """w[N][K] -> (q[N][K] uint8, s[N/128][K/128] float32)."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((_scales(N), _scales(K)), dtype=torch.float32, device=w.device)
    fp8q_quant_w_128x128(w, q, s, stream)
    return q, s


def retile_1x128_to_128x1(q, s, stream=None):
    """Stored 1x128 tiles q[T][C] (scales s[C/128][T]) -> (qT[C][T], sT[T/128][C])."""
    T, C = q.shape
    qT = torch.empty((C, T), dtype=torch.uint8, device=q.device)
    sT = torch.empty((_scales(T), C), dtype=torch.float32, device=q.device)
    fp8q_retile_1x128_to_128x1(q, s, qT, sT, stream)
    return qT, sT


def transpose_w_128x128(q, s, stream=None):
    """q[N][K], s[N/128][K/128] -> (qT[K][N], sT[K/128][N/128])."""
    N, K = q.shape
    qT = torch.empty((K, N), dtype=torch.uint8, device=q.device)
    sT = torch.empty((_scales(K), _scales(N)), dtype=torch.float32, device=q.device)
    fp8q_transpose_w_128x128(q, s, qT, sT, stream)
    return qT, sT


def gemm(A8, sA, B8, sB, out_dtype=torch.bfloat16, bscale=BSCALE_BLOCK128, stream=None,
         stream_k=True):
    """C[M][N] = dequant(A8) @ dequant(B8)^T (stream-K over all SMs unless
    stream_k=False)."""
    C = torch.empty((A8.shape[0], B8.shape[0]), dtype=out_dtype, device=A8.device)
    ws = workspace(A8.device, stream) if stream_k else None
    fp8q_gemm_ws(A8, sA, B8, sB, C, bscale, ws, stream)
    return C


def gemm_quant_a(A, B8, sB, out_dtype=torch.bfloat16, emit=True, stream=None, stream_k=True):
    """C = quant_1x128(A) @ dequant(B8)^T with the quantization inside the GEMM.
    Returns C, or (C, A8, sA) when emit is true."""
    M, K = A.shape
    C = torch.empty((M, B8.shape[0]), dtype=out_dtype, device=A.device)
    A8 = sA = None
    if emit:
        A8 = torch.empty((M, K), dtype=torch.uint8, device=A.device)
        sA = torch.empty((_scales(K), M), dtype=torch.float32, device=A.device)
    ws = workspace(A.device, stream) if stream_k else None
    fp8q_gemm_quant_a(A, B8, sB, C, A8, sA, ws, stream)
    return (C, A8, sA) if emit else C


def gemm_grouped(A8, sA, B8, sB, m_offsets, out_dtype=torch.bfloat16, stream=None,
                 stream_k=True):
    """Grouped GEMM; rows outside every group are left unwritten (uninitialized)."""
    C = torch.empty((A8.shape[0], B8.shape[1]), dtype=out_dtype, device=A8.device)
    ws = workspace(A8.device, stream) if stream_k else None
    fp8q_gemm_grouped_ws(A8, sA, B8, sB, C, m_offsets, ws, stream)
    return C
