"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and nothing else: it holds none of the
quantization or GEMM arithmetic. Both the CUDA path and the CPU oracle are fed
from it.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", 2014) used counter-style -- draw i of stream ``seed`` is
mix64(seed + (i + 1) * 0x9E3779B97F4A7C15) -- so any slice can be produced
independently. Uniforms in (0, 1] take the top 53 bits; normals come from the
Box-Muller transform on consecutive uniform pairs. Values are scaled by sigma,
selected "outlier channels" (K-columns, chosen by a seeded partial
Fisher-Yates shuffle) are multiplied by a factor, and the result is rounded
fp64 -> fp32 -> bf16 (round to nearest even, via torch's CPU cast).

Channel-structured outliers follow the sources' description of LLM
activations: a handful of channels one or two orders of magnitude larger than
the rest ("Low precision: FP8, FP4, and microscaling", outlier paragraph after
the quantize listing; "FP8 Serving" guide, "Things to try").
"""
from __future__ import annotations

import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 23

SEED_X, SEED_W, SEED_X_OUTLIERS, SEED_W_OUTLIERS = 0, 1, 2, 3


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, start: int, n: int) -> np.ndarray:
    z = splitmix64(seed, start, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """n standard normals (fp64) from stream ``seed``."""
    out = np.empty(n, dtype=np.float64)
    for e0 in range(0, n, 2 * _CHUNK):
        e1 = min(n, e0 + 2 * _CHUNK)
        out[e0:e1] = _normal_slice(seed, e0, e1 - e0)
    return out


def outlier_channels(seed: int, k: int, count: int) -> np.ndarray:
    """``count`` distinct indices in [0, k) by a seeded partial Fisher-Yates shuffle (sorted)."""
    count = max(0, min(int(count), k))
    perm = np.arange(k, dtype=np.int64)
    draws = splitmix64(seed, 0, count)
    for i in range(count):
        j = i + int(draws[i] % np.uint64(k - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:count])


def outlier_count(frac: float, k: int) -> int:
    """round(frac * k): 0.5% of 8192 -> 41, of 7168 -> 36; 1% of 4096 -> 41."""
    return int(math.floor(frac * k + 0.5))


def bf16_matrix(rows: int, cols: int, sigma: float, seed: int, outlier_seed: int | None = None,
                outlier_frac: float = 0.0, outlier_factor: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of a [rows, cols] sigma * N(0,1) matrix with outlier columns."""
    import torch

    n = rows * cols
    out = np.empty(n, dtype=np.uint16)
    mult = None
    if outlier_seed is not None and outlier_frac > 0.0:
        ch = outlier_channels(outlier_seed, cols, outlier_count(outlier_frac, cols))
        mult = np.ones(cols, dtype=np.float64)
        mult[ch] = outlier_factor
    step = (_CHUNK // (2 * cols) + 1) * 2 * cols if cols else max(n, 1)
    for e0 in range(0, n, step):
        e1 = min(n, e0 + step)
        z = _normal_slice(seed, e0, e1 - e0) * sigma
        if mult is not None:
            z = (z.reshape(-1, cols) * mult[None, :]).ravel()
        f32 = torch.from_numpy(z.astype(np.float32))
        out[e0:e1] = f32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out.reshape(rows, cols)


def _normal_slice(seed: int, e0: int, n: int) -> np.ndarray:
    """Elements [e0, e0+n) of the stream that ``normal(seed, .)`` produces (e0 even)."""
    assert e0 % 2 == 0
    pairs = (n + 1) // 2
    u = uniform01(seed, e0, 2 * pairs)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = (2.0 * math.pi) * u[1::2]
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z[:n]


# ----------------------------------------------------------------- workloads
# Shapes and distributions of the sources' workloads (DeepSeek-V3-style FP8
# linear layers; decode, prefill, MX and a quantizer sweep).
def tiny():
    """X [128x512] ~N(0,1), W [256x512] ~N(0,0.02); seeds 0 and 1."""
    return bf16_matrix(128, 512, 1.0, SEED_X), bf16_matrix(256, 512, 0.02, SEED_W)


def decode_x(m: int, k: int = 7168):
    return bf16_matrix(m, k, 1.0, SEED_X, SEED_X_OUTLIERS, 0.005, 50.0)


def decode_w(n: int = 18432, k: int = 7168):
    return bf16_matrix(n, k, 0.02, SEED_W)


def prefill_x(m: int = 4096, k: int = 4096):
    return bf16_matrix(m, k, 1.0, SEED_X, SEED_X_OUTLIERS, 0.01, 30.0)


def prefill_w(n: int = 14336, k: int = 4096):
    return bf16_matrix(n, k, 0.02, SEED_W)


def mx_x(m: int = 8192, k: int = 8192):
    return bf16_matrix(m, k, 1.0, SEED_X, SEED_X_OUTLIERS, 0.005, 50.0)


def mx_w(n: int = 8192, k: int = 8192):
    return bf16_matrix(n, k, 1.0, SEED_W, SEED_W_OUTLIERS, 0.005, 50.0)


def sweep_x(rows: int = 16384, cols: int = 8192):
    return bf16_matrix(rows, cols, 1.0, SEED_X, SEED_X_OUTLIERS, 0.005, 100.0)
