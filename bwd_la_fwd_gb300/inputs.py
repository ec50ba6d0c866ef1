"""Seeded synthetic inputs for linear attention (numpy only; none of the method's arithmetic).

Recipe: ``numpy.random.default_rng(seed)`` draws Q, K, V, dO in that order, each as float64
[B, H, N, D] standard normals; Q and K are divided by sqrt(D), so that q . k has standard deviation
1/sqrt(D), while V and dO stay N(0, 1).  Each tensor is then rounded to the storage type: float32 by
round-to-nearest-even, bf16 by round-to-nearest-even from that float32 value.  Multi-layer workloads
draw layer 0, 1, ... in order from one generator.  The oracle and the CUDA path both consume exactly
these rounded values (the oracle after an exact widening to float64).

The shapes are those of the paper's standalone measurements (B=4, H=16, D=128, N swept; N=4096, D
swept; "Transformer Based Linear Attention with Optimized GPU Kernel Implementation", sciencestack.ai
page, Figures 2 and 3).  They are synthetic stand-ins: no dataset is used.
"""
from __future__ import annotations

import numpy as np

TENSORS = ("Q", "K", "V", "dO")
DTYPES = ("f32", "bf16")


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a stored tensor (float32 array, or uint16 bf16 bits)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _draw(rng: np.random.Generator, shape, scale: float, dtype: str, chunk: int) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    done = 0
    while done < n:
        m = min(chunk, n - done)
        x = rng.standard_normal(m)  # float64
        if scale != 1.0:
            x = x * scale
        x32 = x.astype(np.float32)
        out[done:done + m] = f32_to_bf16_bits(x32) if dtype == "bf16" else x32
        done += m
    return out.reshape(shape)


def generate(B: int, H: int, N: int, D: int, seed: int, dtype: str = "bf16", layers: int = 1,
             chunk: int = 1 << 22):
    """Draw the inputs of ``layers`` independent layers from one generator.

    Returns a dict {"Q","K","V","dO"} of stored arrays [B,H,N,D] (float32, or uint16 bf16 bits) when
    ``layers == 1``, else a list of such dicts.  Drawing in chunks gives the same values as one draw.
    """
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}")
    rng = np.random.default_rng(seed)
    shape = (B, H, N, D)
    qk_scale = 1.0 / np.sqrt(D)
    out = []
    for _ in range(layers):
        t = {}
        for name in TENSORS:
            t[name] = _draw(rng, shape, qk_scale if name in ("Q", "K") else 1.0, dtype, chunk)
        out.append(t)
    return out[0] if layers == 1 else out
