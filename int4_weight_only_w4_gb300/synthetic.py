"""Seeded synthetic inputs for the W4 (INT4 weight-only, group 128) GEMV.

This module only draws random numbers and lays them out in the canonical
storage format; it holds none of the product's arithmetic.  It is the one
piece of code that both the CUDA path (tests, benchmark) and the CPU oracle
consume, so that both see bit-identical inputs.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014, in the form of Vigna's public-domain
``splitmix64.c``), used counter-style: element i (0-based) of a stream with
key k is mix(k + (i + 1) * 0x9E3779B97F4A7C15).  Each tensor has its own
stream, keyed by the seed and the tensor's name, so that tensors are
independent and any slice of a stream can be drawn on its own.

Derived draws:
  * packed weights: the top 32 bits of each draw form one uint32 word, so all
    eight nibbles of every word are independent and uniform on 0..15;
  * zeros: the top 4 bits of a draw (uniform on 0..15), stored as uint8;
  * scales: u = top 53 bits * 2^-53 in [0, 1), lo + (hi - lo) * u in fp64,
    rounded to binary16 (numpy, nearest-even);
  * activations: Box-Muller on two draws u1 in (0, 1], u2 in [0, 1),
    sqrt(-2 ln u1) * cos(2 pi u2) in fp64, rounded to binary32 (numpy) and
    then to bfloat16 (nearest-even on the bit pattern).
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1
GROUP = 128

_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _mix_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * _MUL1) & _MASK
    z = ((z ^ (z >> 27)) * _MUL2) & _MASK
    return z ^ (z >> 31)


def _mix(z: np.ndarray) -> np.ndarray:
    z ^= z >> np.uint64(30)
    z *= np.uint64(_MUL1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_MUL2)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, name: str) -> int:
    """Key of the stream for tensor ``name`` under ``seed``."""
    tag = zlib.crc32(name.encode("utf-8"))
    return _mix_int((int(seed) * GAMMA) ^ (tag * 0xD1B54A32D192ED03))


def _u64_range(key: int, start: int, count: int, out: np.ndarray) -> None:
    with np.errstate(over="ignore"):
        z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z *= np.uint64(GAMMA)
        z += np.uint64(key)
        out[:] = _mix(z)


def u64(seed: int, name: str, count: int, start: int = 0) -> np.ndarray:
    """Draws start .. start+count-1 of the stream for ``name`` (uint64)."""
    key = stream_key(seed, name)
    out = np.empty(count, dtype=np.uint64)
    if count <= _CHUNK:
        _u64_range(key, start, count, out)
        return out
    spans = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]
    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(lambda sp: _u64_range(key, start + sp[0], sp[1],
                                          out[sp[0]:sp[0] + sp[1]]), spans))
    return out


def uniform_words(seed: int, name: str, shape) -> np.ndarray:
    """uint32 words with independent uniform nibbles."""
    n = int(np.prod(shape))
    return (u64(seed, name, n) >> np.uint64(32)).astype(np.uint32).reshape(shape)


def uniform_nibbles(seed: int, name: str, shape) -> np.ndarray:
    """uint8 values uniform on 0..15."""
    n = int(np.prod(shape))
    return (u64(seed, name, n) >> np.uint64(60)).astype(np.uint8).reshape(shape)


def uniform_half(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    """binary16 bit patterns of values uniform on [lo, hi)."""
    n = int(np.prod(shape))
    u = (u64(seed, name, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    v = lo + (hi - lo) * u
    return v.astype(np.float16).view(np.uint16).reshape(shape)


def _f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def normal_bf16(seed: int, name: str, shape) -> np.ndarray:
    """bfloat16 bit patterns of standard normal draws."""
    n = int(np.prod(shape))
    d = u64(seed, name, 2 * n)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return _f32_to_bf16_bits(z.astype(np.float32)).reshape(shape)


@dataclass
class Problem:
    """One W4 GEMV instance in the canonical layout (numpy, host memory)."""
    name: str
    M: int
    K: int
    N: int
    qweight: np.ndarray   # uint32 [N, K/8]
    scales: np.ndarray    # uint16 (binary16 bits) [N, K/128]
    zeros: np.ndarray     # uint8 [N, K/128], values 0..15
    x: np.ndarray         # uint16 (bfloat16 bits) [M, K]

    @property
    def G(self) -> int:
        return self.K // GROUP


def make_weights(name: str, K: int, N: int, seed: int = 0,
                 scale_range=(0.001, 0.02)):
    """(qweight, scales, zeros) for an N x K weight with the given scale range."""
    if K <= 0 or K % GROUP or N <= 0:
        raise ValueError(f"K must be a positive multiple of {GROUP} and N positive")
    G = K // GROUP
    qweight = uniform_words(seed, name + "/qweight", (N, K // 8))
    scales = uniform_half(seed, name + "/scales", (N, G), *scale_range)
    zeros = uniform_nibbles(seed, name + "/zeros", (N, G))
    return qweight, scales, zeros


def make_x(name: str, M: int, K: int, seed: int = 0) -> np.ndarray:
    return normal_bf16(seed, name + "/x", (M, K))


def make_problem(name: str, K: int, N: int, M: int, seed: int = 0,
                 scale_range=(0.001, 0.02)) -> Problem:
    qweight, scales, zeros = make_weights(name, K, N, seed, scale_range)
    return Problem(name, M, K, N, qweight, scales, zeros, make_x(name, M, K, seed))


# ---- the workloads -----------------------------------------------------------
# Shapes of the single-request decode GEMVs this library is measured on.
# (name, K, N, token counts, scale range)
SHAPES = [
    ("single.896x896", 896, 896, (1,), (0.001, 0.02)),
    ("qwen0.5b.qkv", 896, 1152, (1,), (0.001, 0.02)),
    ("qwen0.5b.o", 896, 896, (1,), (0.001, 0.02)),
    ("qwen0.5b.gate_up", 896, 9728, (1,), (0.001, 0.02)),
    ("qwen0.5b.down", 4864, 896, (1,), (0.001, 0.02)),
    ("qwen7b.qkv", 3584, 4608, (1,), (0.001, 0.02)),
    ("qwen7b.o", 3584, 3584, (1,), (0.001, 0.02)),
    ("qwen7b.gate_up", 3584, 37888, (1,), (0.001, 0.02)),
    ("qwen7b.down", 18944, 3584, (1,), (0.001, 0.02)),
    ("27b.up", 5120, 17408, (1, 2, 4, 5, 8), (0.0005, 0.01)),
    ("27b.down", 17408, 5120, (1, 2, 4, 5, 8), (0.0005, 0.01)),
    ("qwen7b.lm_head", 3584, 152064, (1, 8), (0.001, 0.02)),
]

# One decoder layer of the 7B-shape model: the four GEMVs of the layer chain.
LAYER_7B = [("qkv", 3584, 4608), ("o", 3584, 3584), ("gate_up", 3584, 37888),
            ("down", 18944, 3584)]
LAYERS_7B = 28

# One decoder layer of the 0.5B-shape model (hidden 896, intermediate 4864,
# 14 query and 2 key/value heads of 64), which has 24 layers.
LAYER_05B = [("qkv", 896, 1152), ("o", 896, 896), ("gate_up", 896, 9728),
             ("down", 4864, 896)]
LAYERS_05B = 24


def shape(name: str):
    for s in SHAPES:
        if s[0] == name:
            return s
    raise KeyError(name)
