"""Shared helpers for the parity tests: moving seeded numpy inputs to the GPU
and the GEMM tolerance.

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
