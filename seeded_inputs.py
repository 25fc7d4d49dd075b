"""Seeded synthetic inputs for the GEMM workloads.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA
side (tests, bench).  It holds none of the GEMM arithmetic: it only draws
numbers.  Every draw is a pure function of (seed, element index), so the same
seed gives the same matrices on any machine and in any chunking.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), element t of stream ``seed`` being the
splitmix64 output for state ``seed + (t + 1) * 0x9E3779B97F4A7C15``.

Distributions (the pages give no recipe; these are the plainest readings of
the workload descriptions):
  * uniform float in [-1, 1):  2 * (top 24 bits) / 2^24 - 1  (exact in fp32)
  * uniform int8 in [-128, 127]: top 8 bits read as a signed byte
  * standard normal: Box-Muller on two independent 53-bit uniforms
  * bf16: round-to-nearest-even of the fp32 value, kept as uint16 bit patterns
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    t = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + t * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, n: int) -> np.ndarray:
    """n raw 64-bit draws of stream ``seed``."""
    out = np.empty(n, dtype=np.uint64)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = _splitmix64(seed, s, c)
    return out


def uniform_f32(shape, seed: int) -> np.ndarray:
    """Uniform floats on the grid k/2^23 - 1 in [-1, 1)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        top = (_splitmix64(seed, s, c) >> np.uint64(40)).astype(np.float64)
        out[s:s + c] = (top * (2.0 / 16777216.0) - 1.0).astype(np.float32)
    return out.reshape(shape)


def uniform_i8(shape, seed: int) -> np.ndarray:
    """Uniform int8 over the full range [-128, 127]."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = (_splitmix64(seed, s, c) >> np.uint64(56)).astype(np.uint8).view(np.int8)
    return out.reshape(shape)


def small_int_f32(shape, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Integers in [lo, hi] stored as float32 (exact in fp32 and bf16 for |v| <= 256)."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = ((_splitmix64(seed, s, c) >> np.uint64(11)) % span).astype(np.int64) + lo
    return out.reshape(shape)


def normal_f32(shape, seed: int) -> np.ndarray:
    """Standard normal draws (Box-Muller), rounded to float32."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    half = (n + 1) // 2
    for s in range(0, half, _CHUNK):
        c = min(_CHUNK, half - s)
        r = _splitmix64(seed, 2 * s, 2 * c)
        u1 = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
        u2 = (r[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        rad = np.sqrt(-2.0 * np.log(u1))
        ang = 2.0 * np.pi * u2
        z = np.empty(2 * c, dtype=np.float64)
        z[0::2] = rad * np.cos(ang)
        z[1::2] = rad * np.sin(ang)
        lo, hi = 2 * s, min(2 * s + 2 * c, n)
        out[lo:hi] = z[: hi - lo].astype(np.float32)
    return out.reshape(shape)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------------ workloads
def config_seed(index: int, sub: int = 0) -> int:
    """Seed of workload ``index`` (and of its sub-case ``sub``, e.g. one K of a sweep)."""
    return 0x5EED0000 + (index << 8) + sub


def workload(name: str, M: int, N: int, K: int, seed: int):
    """Operands (A, B, C_in, alpha, beta, dtype) of one named workload recipe.

    Recipes (shapes are the caller's):
      "f32_uniform"       fp32 A, B ~ U[-1,1); C zero; alpha=1, beta=0
      "f32_uniform_beta"  fp32 A, B, C ~ U[-1,1); alpha=1, beta=0.5
      "i8_uniform"        int8 A, B ~ U{-128..127}; C zero (int32); alpha=1, beta=0
      "bf16_normal"       bf16(RNE of N(0,1)) A, B; C zero; alpha=1, beta=0
    """
    if name == "f32_uniform":
        A = uniform_f32((M, K), seed)
        B = uniform_f32((K, N), seed + 1)
        return A, B, np.zeros((M, N), np.float32), 1.0, 0.0, "f32"
    if name == "f32_uniform_beta":
        A = uniform_f32((M, K), seed)
        B = uniform_f32((K, N), seed + 1)
        C = uniform_f32((M, N), seed + 2)
        return A, B, C, 1.0, 0.5, "f32"
    if name == "i8_uniform":
        A = uniform_i8((M, K), seed)
        B = uniform_i8((K, N), seed + 1)
        return A, B, np.zeros((M, N), np.int32), 1, 0, "i8"
    if name == "bf16_normal":
        A = to_bf16_bits(normal_f32((M, K), seed))
        B = to_bf16_bits(normal_f32((K, N), seed + 1))
        return A, B, np.zeros((M, N), np.float32), 1.0, 0.0, "bf16"
    raise KeyError(name)
