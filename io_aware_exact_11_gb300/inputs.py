"""Seeded synthetic inputs for attention workloads.

This module only draws random numbers and rounds them to the storage type.
It holds none of the attention arithmetic, so both the CUDA library's tests
and the float64 oracle can be fed from it.

Recipe: every (tensor, b, h) slice has its own PCG64 stream keyed by
``[seed, tensor_id, b, h]`` and is drawn as float32 i.i.d. N(0, 1) of shape
[rows, d].  A full [B, H, N, d] tensor is the stack of its slices, so any
single head can be regenerated without drawing the whole tensor.  For bf16
workloads the float32 draws are rounded to bf16 (round to nearest, ties to
even); the oracle then reads exactly those rounded values as float64.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "do": 3}


def normal_slice(seed: int, name: str, b: int, h: int, rows: int, d: int) -> np.ndarray:
    """float32 N(0,1) block [rows, d] for one (tensor, b, h) slice."""
    g = np.random.Generator(np.random.PCG64([int(seed), TENSOR_IDS[name], int(b), int(h)]))
    return g.standard_normal((rows, d), dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits (uint16) to float32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities; finite values saturate at ±448), nearest-even.  Returns
    uint8 codes.  Used to build FP8 inputs; the oracle reads them back with
    ``e4m3_bits_to_f32``."""
    x = np.asarray(x, dtype=np.float32)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.minimum(np.abs(x).astype(np.float64), 448.0)
    out = np.zeros(a.shape, dtype=np.uint8)
    # Normal range: exponent e in [-6, 8], value = 2^e · (1 + m/8).
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    step = np.exp2(e - 3)                       # spacing of representable values
    q = np.round(a / step) * step               # np.round is half-to-even
    # Rounding can carry into the next binade; recompute its exponent.
    e2 = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    normal = q >= 2.0 ** -6
    mant = np.where(normal, np.round(q / np.exp2(e2) * 8) - 8, np.round(q / 2.0 ** -9))
    expf = np.where(normal, e2 + 7, 0)
    code = (expf.astype(np.int64) << 3) | mant.astype(np.int64)
    out[...] = np.where(a > 0, code, 0).astype(np.uint8)
    return out | sign


def e4m3_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact value of FP8 E4M3 codes (uint8) as float32 (the NaN code maps to NaN)."""
    u = np.asarray(u, dtype=np.uint8).astype(np.int64)
    s = np.where(u & 0x80, -1.0, 1.0)
    e = (u >> 3) & 0xF
    m = u & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return (s * val).astype(np.float32)


def _threads() -> int:
    return max(1, min(16, len(os.sched_getaffinity(0))))


def normal_tensor(seed: int, name: str, B: int, H: int, N: int, d: int, dtype: str = "bf16") -> np.ndarray:
    """Full [B, H, N, d] tensor built slice by slice.

    dtype "bf16" returns uint16 bf16 bits; "fp32" returns float32.
    """
    if dtype == "bf16":
        out = np.empty((B, H, N, d), dtype=np.uint16)
    elif dtype == "fp32":
        out = np.empty((B, H, N, d), dtype=np.float32)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")

    def fill(bh):
        b, h = divmod(bh, H)
        x = normal_slice(seed, name, b, h, N, d)
        out[b, h] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    if B * H * N * d >= (1 << 22) and B * H > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(B * H)))
    else:
        for bh in range(B * H):
            fill(bh)
    return out


def head_as_f64(seed: int, name: str, b: int, h: int, rows: int, d: int, dtype: str = "bf16") -> np.ndarray:
    """One slice as the float64 values the kernels see (bf16-rounded if bf16)."""
    x = normal_slice(seed, name, b, h, rows, d)
    if dtype == "bf16":
        x = bf16_bits_to_f32(f32_to_bf16_bits(x))
    return x.astype(np.float64)


def as_f64(t: np.ndarray, dtype: str) -> np.ndarray:
    """Host tensor from ``normal_tensor`` widened to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(t).astype(np.float64)
    return np.asarray(t, dtype=np.float64)
