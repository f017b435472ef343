"""Seeded synthetic inputs for the fine-grained FP8 path.

This module is the one piece shared by the CUDA package's tests/benchmark and
the CPU oracle's tests: it draws random tensors and nothing else.  It holds
none of the method's arithmetic (no amax, no scale, no FP8 cast, no GEMM).

Every tensor of a workload gets its own numpy PCG64 stream seeded with
``SeedSequence([seed, tensor_index])``, so any one tensor can be regenerated
alone.  BF16 tensors are drawn in FP32 and rounded to nearest-even BF16; they
are returned as numpy ``uint16`` bit patterns, FP32 tensors as ``float32``.

Workloads (DeepSeek-V3-shaped, per the fine-grained FP8 GEMM description):
  tiny      A[128][512], B[128][512] FP32 N(0,1), 0.1% of entries x50
  forward   A[4096][7168] BF16 N(0,1) with 0.1% x100; W[2048][7168] BF16 N(0, 0.02)
  accum     A[1024][16384], B[1024][16384] BF16 U(-1,1); variant "positive": U(0,1)
  wgrad     dY[8192][7168], X[8192][2048] BF16 N(0,1), 0.1% x100 each
  grouped   32 experts, token counts ~ Multinomial(16384, p_i ~ i^-1.1) rounded
            up to multiples of 128; A[sum M_e][7168] BF16 N(0,1) with 0.1% x100;
            W[32][2048][7168] BF16 N(0, 0.02)
  backward  the forward workload's A and W plus dY[4096][2048] BF16 N(0,1), 0.1% x100
  mlp_down  gate_up[4096][2*2048] BF16 N(0,1), 0.1% x100 (gate | up halves of the
            up-projection output); W2[7168][2048] BF16 N(0, 0.02)
  forward_norm  the forward workload with its activations normalized first:
            X[4096][7168] BF16 N(0,1), 0.1% x100 (un-normalized), RMSNorm weight
            g[7168] BF16 N(1, 0.1), W[2048][7168] BF16 N(0, 0.02)
Outliers: floor(0.1% of the entries) positions drawn uniformly without
replacement; the value already there is multiplied by the factor.
"""
import numpy as np
import torch

GROUP = 128

CONFIG_NAMES = ("tiny", "forward", "accum", "wgrad", "grouped", "backward", "mlp_down",
                "forward_norm")


def rng_for(seed: int, tensor_index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_index])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 to nearest-even BF16; return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _outliers(x: np.ndarray, rng: np.random.Generator, frac: float, mult: float) -> None:
    n = x.size
    k = int(n * frac)
    if k <= 0 or mult == 1.0:
        return
    idx = rng.choice(n, size=k, replace=False)
    flat = x.reshape(-1)
    flat[idx] *= np.float32(mult)


def gaussian(shape, rng, std=1.0, outlier_frac=0.0, outlier_mult=1.0, bf16=True):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    _outliers(x, rng, outlier_frac, outlier_mult)
    return to_bf16_bits(x) if bf16 else x


def uniform(shape, rng, lo=-1.0, hi=1.0, bf16=True):
    x = rng.random(size=shape, dtype=np.float32)
    x = x * np.float32(hi - lo) + np.float32(lo)
    return to_bf16_bits(x) if bf16 else x


def zipf_group_sizes(rng, tokens=16384, groups=32, s=1.1, align=GROUP):
    """Per-expert row counts: Multinomial(tokens, p_i ~ i^-s), each rounded up
    to a multiple of `align` (an expert with no tokens keeps 0 rows)."""
    p = np.arange(1, groups + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    counts = rng.multinomial(tokens, p)
    sizes = ((counts + align - 1) // align) * align
    return sizes.astype(np.int64)


def offsets_from_sizes(sizes) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(sizes, dtype=np.int64))]).astype(np.int64)


def make(name: str, seed: int = 0, variant: str = "", scale_down: int = 1):
    """Tensors of one workload.  ``scale_down`` > 1 divides the row counts
    (M, N, T, tokens) by that factor -- same distributions, smaller problem --
    for quick parity runs; K stays as named unless the workload says otherwise."""
    d = int(scale_down)
    if name == "tiny":
        return {
            "A": gaussian((128, 512), rng_for(seed, 0), 1.0, 0.001, 50.0, bf16=False),
            "B": gaussian((128, 512), rng_for(seed, 1), 1.0, 0.001, 50.0, bf16=False),
            "out": "f32",
        }
    if name == "forward":
        return {
            "A": gaussian((4096 // d, 7168), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "W": gaussian((2048 // d, 7168), rng_for(seed, 1), 0.02),
            "out": "bf16",
        }
    if name == "accum":
        lo = 0.0 if variant == "positive" else -1.0
        return {
            "A": uniform((1024 // d, 16384), rng_for(seed, 0), lo, 1.0),
            "B": uniform((1024 // d, 16384), rng_for(seed, 1), lo, 1.0),
            "out": "f32",
        }
    if name == "wgrad":
        return {
            "dY": gaussian((8192 // d, 7168 // d), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "X": gaussian((8192 // d, 2048 // d), rng_for(seed, 1), 1.0, 0.001, 100.0),
            "out": "f32",
        }
    if name == "backward":
        # the backward data path of the forward workload: its A and W (same
        # streams as "forward") plus an output gradient dY[M][N]
        return {
            "A": gaussian((4096 // d, 7168), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "W": gaussian((2048 // d, 7168), rng_for(seed, 1), 0.02),
            "dY": gaussian((4096 // d, 2048 // d), rng_for(seed, 2), 1.0, 0.001, 100.0),
            "out": "bf16",
        }
    if name == "grouped":
        sizes = zipf_group_sizes(rng_for(seed, 2), tokens=16384 // d)
        offs = offsets_from_sizes(sizes)
        mtot = int(offs[-1])
        return {
            "A": gaussian((mtot, 7168), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "W": gaussian((32, 2048 // d, 7168), rng_for(seed, 1), 0.02),
            "m_offsets": offs,
            "out": "bf16",
        }
    if name == "forward_norm":
        g = (1.0 + 0.1 * rng_for(seed, 2).standard_normal(7168)).astype(np.float32)
        return {
            "X": gaussian((4096 // d, 7168), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "g": to_bf16_bits(g),
            "W": gaussian((2048 // d, 7168), rng_for(seed, 1), 0.02),
            "out": "bf16",
        }
    if name == "mlp_down":
        # SwiGLU MLP down projection: the gate and up halves of the up
        # projection's output side by side, and the down-projection weight
        return {
            "gate_up": gaussian((4096 // d, 2 * 2048), rng_for(seed, 0), 1.0, 0.001, 100.0),
            "W2": gaussian((7168 // d, 2048), rng_for(seed, 1), 0.02),
            "out": "bf16",
        }
    raise ValueError("unknown workload %r" % name)
