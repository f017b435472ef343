"""Shared helpers for the parity tests: moving seeded numpy inputs to the GPU,
the GEMM tolerance, and the check of the fused FP32-evaluated casts.

Tolerance (the bar stated for this path): FP32 output
|C - C_ref| <= 1e-5 * sum_k |a_k b_k|; BF16 output adds one BF16 unit in the
last place of C_ref (the output is rounded once, to nearest even).
"""
import numpy as np
import torch

GEMM_RTOL_ABS = 1e-5


def to_dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are BF16 bit patterns."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def gemm_bound(Cabs: np.ndarray, Cref: np.ndarray, bf16_out: bool) -> np.ndarray:
    b = GEMM_RTOL_ABS * Cabs
    if bf16_out:
        b = b + bf16_ulp(Cref)
    return b


def assert_gemm_close(C_gpu: np.ndarray, Cref: np.ndarray, Cabs: np.ndarray, bf16_out: bool,
                      what=""):
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    err = np.abs(C_gpu - Cref)
    bound = gemm_bound(Cabs, Cref, bf16_out)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = ["%s: gpu=%r ref=%r abs=%r bound=%r" % (
            tuple(i), C_gpu[tuple(i)], Cref[tuple(i)], Cabs[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError("%s: %d / %d entries out of tolerance; first: %s" % (
            what, int(bad.sum()), bad.size, "; ".join(details)))
    return float(np.max(err / np.maximum(Cabs, 1e-300)))


def cpu(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def exact_scaled_1x128(h: np.ndarray) -> np.ndarray:
    """h (FP64, [M][K], K a multiple of 128) -> h * inv of its 1x128 tile, inv
    as the 1x128 rule makes it from the FP32-rounded values (amax 0 -> 1;
    an overflowing inverse clamped to the largest float)."""
    M, K = h.shape
    h32 = h.astype(np.float32)
    amax = np.abs(h32).reshape(M, K // 128, 128).max(axis=2)
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.where(amax == 0, np.float32(1.0), np.float32(448.0) / amax).astype(np.float32)
    inv = np.where(np.isinf(inv), np.finfo(np.float32).max, inv)
    return h * np.repeat(inv.astype(np.float64), 128, axis=1)


def check_fused_1x128(oracle, q_gpu, s_gpu, h, q_o, s_o, h_rel, s_rel, what):
    """A fused operator + 1x128 cast evaluated in FP32 against the oracle's
    exact operator (h, FP64) and its quantization (q_o, s_o):
      * scales within s_rel relative;
      * every code the round-to-nearest-even E4M3 encoding of some value
        within h_rel relative of the exact scaled value h * inv (at a rounding
        boundary either neighbour passes, anywhere else only one code);
      * at least 99.9 % of the codes identical to the oracle's."""
    s_gpu = np.asarray(s_gpu, np.float64)
    rel = np.abs(s_gpu / np.asarray(s_o, np.float64) - 1.0)
    assert rel.max() <= s_rel, "%s: scale off by %.3g relative" % (what, rel.max())
    y = exact_scaled_1x128(h)
    ends = [oracle.e4m3_decode(oracle.e4m3_encode((y * (1.0 + e)).astype(np.float32)))
            for e in (-h_rel, h_rel)]
    lo, hi = np.minimum(ends[0], ends[1]), np.maximum(ends[0], ends[1])
    d = oracle.e4m3_decode(np.asarray(q_gpu))
    bad = np.argwhere((d < lo) | (d > hi))
    assert bad.size == 0, "%s: %d codes outside the interval, first at %s (gpu %r, allowed %r..%r)" % (
        what, len(bad), tuple(bad[0]), d[tuple(bad[0])], lo[tuple(bad[0])], hi[tuple(bad[0])])
    same = np.mean(np.asarray(q_gpu) == q_o)
    assert same >= 0.999, "%s: only %.4f of codes equal the oracle's" % (what, same)


GUARD_BYTES = 4096          # guard band on each side (keeps 16-byte alignment)
SENTINEL = 0xA7


class Guarded:
    """A CUDA output tensor of `shape` and `dtype` placed inside a larger byte
    buffer whose guard bands, GUARD_BYTES before and after it, hold a sentinel
    byte.  check() asserts that a kernel wrote nothing outside the tensor (the
    stand-in for a memory checker on the GPU)."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        es = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * es
        self.buf = torch.full((2 * GUARD_BYTES + self.nbytes,), SENTINEL, dtype=torch.uint8,
                              device=device)
        self.t = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(tuple(shape))
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what=""):
        torch.cuda.synchronize()
        head = self.buf[:GUARD_BYTES]
        tail = self.buf[GUARD_BYTES + self.nbytes:]
        nh = int((head != SENTINEL).sum().item())
        nt = int((tail != SENTINEL).sum().item())
        assert nh == 0 and nt == 0, "%s: %d bytes written before and %d after the buffer" % (
            what, nh, nt)
