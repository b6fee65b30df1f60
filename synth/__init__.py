"""Seeded synthetic inputs for the attention workloads.

This module is the one piece of code shared by the FP64 oracle side and the
CUDA side of the test suite.  It draws numbers and rounds them to bfloat16; it
holds none of the attention arithmetic.

Generator (counter based, so any element can be drawn on its own):

* ``u64(seed, i)`` is the i-th output of the splitmix64 sequence started at
  ``seed``: the state after ``i + 1`` additions of the golden-ratio increment
  0x9E3779B97F4A7C15, passed through the splitmix64 finaliser (xor-shift 30,
  multiply 0xBF58476D1CE4E5B9, xor-shift 27, multiply 0x94D049BB133111EB,
  xor-shift 31).
* ``uniform(seed, i) = (u64(seed, i) >> 11) * 2**-53`` lies in [0, 1).
* Normal number ``n`` of a stream comes from the Box-Muller transform of the
  uniform pair at counters ``2*(n//2)`` and ``2*(n//2) + 1``:
  ``r = sqrt(-2 ln(1 - u_a))``, ``t = 2 pi u_b``; even ``n`` takes ``r cos t``,
  odd ``n`` takes ``r sin t``.
* bfloat16 values are the FP32 rounding of that FP64 normal, then rounded to
  bfloat16 with round-to-nearest-even.

A workload draws its tensors from one stream (seed 0 unless stated) in the
order Q, K, V, dO; each tensor starts where the previous one ended.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """The ``counters``-th outputs (uint64 array) of splitmix64 seeded by ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (counters.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(seed: int, counters: np.ndarray) -> np.ndarray:
    """Uniform FP64 numbers in [0, 1) at the given counters."""
    return (splitmix64(seed, counters) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_f64(seed: int, start: int, count: int) -> np.ndarray:
    """Normals ``start .. start+count-1`` of the stream (``start`` must be even)."""
    if start % 2:
        raise ValueError("normal streams are addressed in Box-Muller pairs; start must be even")
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        pairs = np.arange(start // 2 + p0, start // 2 + p1, dtype=np.uint64)
        ua = uniform(seed, pairs * np.uint64(2))
        ub = uniform(seed, pairs * np.uint64(2) + np.uint64(1))
        r = np.sqrt(-2.0 * np.log1p(-ua))
        t = (2.0 * math.pi) * ub
        blk = np.empty(2 * (p1 - p0), dtype=np.float64)
        blk[0::2] = r * np.cos(t)
        blk[1::2] = r * np.sin(t)
        n0 = 2 * p0
        n1 = min(count, 2 * p1)
        out[n0:n1] = blk[: n1 - n0]
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to FP32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_bits(seed: int, start: int, shape) -> np.ndarray:
    """A tensor of N(0,1) draws rounded to bfloat16 (uint16 bit patterns)."""
    count = int(np.prod(shape))
    return f32_to_bf16_bits(normal_f64(seed, start, count).astype(np.float32)).reshape(shape)


@dataclass(frozen=True)
class AttentionShape:
    B: int
    H: int
    N: int
    d_qk: int
    d_v: int


def attention_inputs(shape: AttentionShape, seed: int = 0, with_do: bool = True) -> dict:
    """Q, K, V (and dO) as bfloat16 bit patterns, layout [B, H, N, d], drawn in that order."""
    B, H, N, dqk, dv = shape.B, shape.H, shape.N, shape.d_qk, shape.d_v
    sizes = [("q", (B, H, N, dqk)), ("k", (B, H, N, dqk)), ("v", (B, H, N, dv))]
    if with_do:
        sizes.append(("do", (B, H, N, dv)))
    out = {}
    pos = 0
    for name, shp in sizes:
        out[name] = normal_bf16_bits(seed, pos, shp)
        pos += int(np.prod(shp))
        pos += pos % 2
    return out


# ----------------------------------------------------------------------------
# The same generator evaluated with torch tensors (on a GPU for large inputs).
# Identical definition; int64 arithmetic wraps like uint64 and right shifts are
# masked to be logical.  libm differences between devices can move an FP64
# normal by an ulp, which after rounding to bfloat16 almost never shows; each
# test therefore draws its inputs once and hands the same bits to both sides.
def _as_i64(x: int) -> int:
    x &= 0xFFFFFFFFFFFFFFFF
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr(t, k: int):
    return (t >> k) & ((1 << (64 - k)) - 1)


def normal_bf16_torch(seed: int, start: int, shape, device="cuda"):
    """Like ``normal_bf16_bits`` but returns a torch.bfloat16 tensor on ``device``."""
    import torch

    if start % 2:
        raise ValueError("start must be even")
    count = int(np.prod(shape))
    npairs = (count + 1) // 2
    out = torch.empty(2 * npairs, dtype=torch.float64, device=device)
    g, m1, m2, sd = _as_i64(0x9E3779B97F4A7C15), _as_i64(0xBF58476D1CE4E5B9), _as_i64(0x94D049BB133111EB), _as_i64(seed)
    chunk = 1 << 24
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        pairs = torch.arange(start // 2 + p0, start // 2 + p1, dtype=torch.int64, device=device)
        u = []
        for off in (0, 1):
            z = (pairs * 2 + off + 1) * g + sd
            z = (z ^ _lsr(z, 30)) * m1
            z = (z ^ _lsr(z, 27)) * m2
            z = z ^ _lsr(z, 31)
            u.append(_lsr(z, 11).to(torch.float64) * (2.0 ** -53))
        r = torch.sqrt(-2.0 * torch.log1p(-u[0]))
        t = (2.0 * math.pi) * u[1]
        out[2 * p0:2 * p1:2] = r * torch.cos(t)
        out[2 * p0 + 1:2 * p1:2] = r * torch.sin(t)
    return out[:count].to(torch.float32).to(torch.bfloat16).reshape(shape)


def attention_inputs_torch(shape: AttentionShape, seed: int = 0, with_do: bool = True, device="cuda") -> dict:
    """Q, K, V (and dO) as torch.bfloat16 tensors, same stream layout as ``attention_inputs``."""
    B, H, N, dqk, dv = shape.B, shape.H, shape.N, shape.d_qk, shape.d_v
    sizes = [("q", (B, H, N, dqk)), ("k", (B, H, N, dqk)), ("v", (B, H, N, dv))]
    if with_do:
        sizes.append(("do", (B, H, N, dv)))
    out = {}
    pos = 0
    for name, shp in sizes:
        out[name] = normal_bf16_torch(seed, pos, shp, device)
        pos += int(np.prod(shp))
        pos += pos % 2
    return out


# ----------------------------------------------------------------------------
# Decode-shaped workloads: N_q queries against N_k keys (split-KV forward).
@dataclass(frozen=True)
class DecodeShape:
    B: int
    H: int
    N_q: int
    N_k: int
    d_qk: int
    d_v: int


def _decode_sizes(shape: DecodeShape):
    B, H = shape.B, shape.H
    return [("q", (B, H, shape.N_q, shape.d_qk)), ("k", (B, H, shape.N_k, shape.d_qk)),
            ("v", (B, H, shape.N_k, shape.d_v))]


def decode_inputs(shape: DecodeShape, seed: int = 0) -> dict:
    """Q [B,H,N_q,d_qk], K [B,H,N_k,d_qk], V [B,H,N_k,d_v] as bfloat16 bit
    patterns, drawn in that order from one stream (as ``attention_inputs``)."""
    out = {}
    pos = 0
    for name, shp in _decode_sizes(shape):
        out[name] = normal_bf16_bits(seed, pos, shp)
        pos += int(np.prod(shp))
        pos += pos % 2
    return out


def decode_inputs_torch(shape: DecodeShape, seed: int = 0, device="cuda") -> dict:
    """``decode_inputs`` as torch.bfloat16 tensors on ``device``."""
    out = {}
    pos = 0
    for name, shp in _decode_sizes(shape):
        out[name] = normal_bf16_torch(seed, pos, shp, device)
        pos += int(np.prod(shp))
        pos += pos % 2
    return out
