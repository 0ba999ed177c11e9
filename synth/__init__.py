"""Seeded synthetic inputs for the EXL3 trellis linear.

This module is the only code shared by the CPU oracle and the CUDA path. It
holds no arithmetic of the method itself: it draws random code words, random
+-1 sign vectors and Gaussian activations, nothing else.

Recipe (every draw uses numpy's PCG64 seeded by ``SeedSequence([seed, stream])``
so each quantity has its own independent stream):

* codes  (stream 1): uniform random uint32 words, ``TK x (TN*8*bits)``. Every
  bit string is a valid tail-biting trellis code, so uniform words are uniform
  codes.
* suh    (stream 2): uniform +-1, length K, stored as FP16.
* svh    (stream 3): uniform +-1, length N, stored as FP16.
* x      (stream 4): N(0,1) drawn in FP64, rounded to FP16 (or BF16), R x K.

Group members draw from streams offset by ``16 * member`` so q, k and v get
distinct codes and sign vectors.
"""
from __future__ import annotations

import numpy as np

STREAM_CODES, STREAM_SUH, STREAM_SVH, STREAM_X = 1, 2, 3, 4


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def codes(seed: int, K: int, N: int, bits: int, member: int = 0) -> np.ndarray:
    """Uniform random trellis words, shape (K//16, (N//16)*8*bits), uint32."""
    if K % 16 or N % 16 or not (1 <= bits <= 8):
        raise ValueError("K, N must be multiples of 16 and 1 <= bits <= 8")
    g = _rng(seed, STREAM_CODES + 16 * member)
    return g.integers(0, 1 << 32, size=(K // 16, (N // 16) * 8 * bits), dtype=np.uint64).astype(np.uint32)


def signs(seed: int, n: int, stream: int, member: int = 0) -> np.ndarray:
    """Uniform +-1 vector as float16."""
    g = _rng(seed, stream + 16 * member)
    return np.where(g.integers(0, 2, size=n) == 1, 1.0, -1.0).astype(np.float16)


def suh(seed: int, K: int, member: int = 0) -> np.ndarray:
    return signs(seed, K, STREAM_SUH, member)


def svh(seed: int, N: int, member: int = 0) -> np.ndarray:
    return signs(seed, N, STREAM_SVH, member)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def activations(seed: int, rows: int, K: int, dtype: str = "f16") -> np.ndarray:
    """x ~ N(0,1), rows x K. Returns float16 for 'f16', uint16 bf16 bits for 'bf16'."""
    g = _rng(seed, STREAM_X)
    a = g.standard_normal(size=(rows, K))
    if dtype == "f16":
        return a.astype(np.float16)
    if dtype == "bf16":
        # FP64 -> FP32 is exact for the rounding decision here only up to the
        # double rounding FP64->FP32->BF16; the value drawn is arbitrary anyway.
        return f32_to_bf16_bits(a.astype(np.float32))
    raise ValueError(dtype)


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 copy of an f16 array or of bf16 bit patterns."""
    return x.astype(np.float64) if dtype == "f16" else bf16_bits_to_f64(x)
