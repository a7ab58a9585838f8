"""CPU oracle for the weight-only INT4 (group 128) matrix-vector product.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
(``int4_weight_only_w4_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``w4_oracle.c`` (plain single-threaded C, fp64 dot
products; see its header for the passages it follows).  This module only
compiles it with gcc and marshals numpy arrays into it with ctypes.

Array conventions (all numpy, C-contiguous):
  qweight  uint32 [N, K/8]   nibble j of word w holds k = 8w + j (bits 4j..4j+3)
  scales   uint16 [N, K/128] binary16 bit patterns
  zeros    uint8  [N, K/128]
  x        uint16 [M, K]     bfloat16 bit patterns
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libw4oracle.so")
_lib = None
_OMP_SRC = os.path.join(_HERE, "w4_cpu_omp.c")
_OMP_PATH = os.path.join(_HERE, "libw4cpu_omp.so")
_omp = None

GROUP = 128


def build(force: bool = False) -> str:
    """Compile w4_oracle.c into libw4oracle.so next to it (gcc, no fast-math,
    no multiply-add contraction).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_omp(force: bool = False) -> str:
    """Compile the OpenMP CPU baseline (w4_cpu_omp.c) into libw4cpu_omp.so."""
    if (not force and os.path.exists(_OMP_PATH)
            and os.path.getmtime(_OMP_PATH) >= os.path.getmtime(_OMP_SRC)):
        return _OMP_PATH
    tmp = _OMP_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _OMP_SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OMP_PATH)
    return _OMP_PATH


def _load_omp():
    global _omp
    if _omp is None:
        lib = ctypes.CDLL(build_omp())
        lib.w4c_threads.restype = ctypes.c_int
        lib.w4c_threads.argtypes = []
        lib.w4c_gemv_f64.restype = None
        lib.w4c_gemv_f64.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
        _omp = lib
    return _omp


def omp_threads() -> int:
    """Threads the OpenMP CPU baseline uses (all host cores unless limited)."""
    return int(_load_omp().w4c_threads())


def gemv_f64_omp(qweight, scales, zeros, x, M: int, K: int, N: int):
    """The same y[M, N] as gemv_f64, computed with the rows spread over all
    host cores (CPU baseline for timing; bit-identical to gemv_f64)."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, N)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.shape != (M, K):
        raise ValueError("x must be [M, K]")
    y = np.empty((M, N), dtype=np.float64)
    _load_omp().w4c_gemv_f64(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), M, K, N,
                             _ptr(y))
    return y


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.w4o_half_to_double.restype = ctypes.c_double
    lib.w4o_half_to_double.argtypes = [ctypes.c_uint16]
    lib.w4o_bf16_to_double.restype = ctypes.c_double
    lib.w4o_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.w4o_double_to_half_rne.restype = ctypes.c_uint16
    lib.w4o_double_to_half_rne.argtypes = [ctypes.c_double]
    lib.w4o_float_to_bf16_rne.restype = ctypes.c_uint16
    lib.w4o_float_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.w4o_float_to_bf16_rne_array.restype = None
    lib.w4o_float_to_bf16_rne_array.argtypes = [P, P, ctypes.c_int64]
    lib.w4o_dequant_f32.restype = None
    lib.w4o_dequant_f32.argtypes = [P, P, P, I, I, P]
    lib.w4o_dequant_f16.restype = None
    lib.w4o_dequant_f16.argtypes = [P, P, P, I, I, P]
    lib.w4o_gemv_f64.restype = None
    lib.w4o_gemv_f64.argtypes = [P, P, P, P, I, I, I, P, P]
    lib.w4o_gemv_rows_f64.restype = None
    lib.w4o_gemv_rows_f64.argtypes = [P, P, P, P, I, I, P, I, P, P]
    lib.w4o_gemv_swiglu_f64.restype = None
    lib.w4o_gemv_swiglu_f64.argtypes = [P, P, P, P, I, I, I, P]
    lib.w4o_quantize.restype = None
    lib.w4o_quantize.argtypes = [P, I, I, I, P, P, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(qweight, scales, zeros, K, N):
    if K <= 0 or K % GROUP or N <= 0:
        raise ValueError(f"bad shape K={K} N={N}")
    G = K // GROUP
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    zeros = np.ascontiguousarray(zeros, dtype=np.uint8)
    if qweight.shape != (N, K // 8) or scales.shape != (N, G) or zeros.shape != (N, G):
        raise ValueError("qweight/scales/zeros shapes do not match K, N")
    return qweight, scales, zeros


# ---- scalar number-format helpers (exposed for the pin tests) --------------

def half_to_double(bits: int) -> float:
    return _load().w4o_half_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().w4o_bf16_to_double(int(bits))


def double_to_half_rne(v: float) -> int:
    return int(_load().w4o_double_to_half_rne(float(v)))


def float_to_bf16_rne(v: float) -> int:
    return int(_load().w4o_float_to_bf16_rne(float(v)))


def bf16_rne(y: np.ndarray) -> np.ndarray:
    """Elementwise fp32 -> bfloat16 bits with the oracle's own rounding."""
    flat = np.ascontiguousarray(np.asarray(y, dtype=np.float32).ravel())
    out = np.empty(flat.shape, dtype=np.uint16)
    _load().w4o_float_to_bf16_rne_array(_ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(y))


# ---- dequantisation and the matrix-vector product ---------------------------

def dequant_f32(qweight, scales, zeros, K: int, N: int) -> np.ndarray:
    """(q - z) * s as float32 [N, K] (exact)."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, N)
    out = np.empty((N, K), dtype=np.float32)
    _load().w4o_dequant_f32(_ptr(qweight), _ptr(scales), _ptr(zeros), K, N, _ptr(out))
    return out


def dequant_f16(qweight, scales, zeros, K: int, N: int) -> np.ndarray:
    """binary16 bits [N, K] of (q - z) * s rounded once to nearest-even."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, N)
    out = np.empty((N, K), dtype=np.uint16)
    _load().w4o_dequant_f16(_ptr(qweight), _ptr(scales), _ptr(zeros), K, N, _ptr(out))
    return out


def gemv_f64(qweight, scales, zeros, x, M: int, K: int, N: int, with_abs: bool = False):
    """y[M, N] = sum_k (q - z) * s * x in fp64.  With ``with_abs`` also returns
    sum_k |(q - z) * s * x| (for rounding-error bounds)."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, N)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.shape != (M, K):
        raise ValueError("x must be [M, K]")
    y = np.empty((M, N), dtype=np.float64)
    yabs = np.empty((M, N), dtype=np.float64) if with_abs else None
    _load().w4o_gemv_f64(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), M, K, N,
                         _ptr(y), _ptr(yabs) if with_abs else None)
    return (y, yabs) if with_abs else y


def gemv_rows_f64(qweight, scales, zeros, x, M: int, K: int, N: int, rows,
                  with_abs: bool = False):
    """The product restricted to output rows ``rows``: y[M, len(rows)]."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, N)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if x.shape != (M, K):
        raise ValueError("x must be [M, K]")
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row index out of range")
    R = rows.size
    y = np.empty((M, R), dtype=np.float64)
    yabs = np.empty((M, R), dtype=np.float64) if with_abs else None
    _load().w4o_gemv_rows_f64(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), M, K,
                              _ptr(rows), R, _ptr(y), _ptr(yabs) if with_abs else None)
    return (y, yabs) if with_abs else y


QUANT_ASYM = 0      # w4o_quantize mode 0: min/max including 0, zero point per group
QUANT_SYM = 1       # mode 1: the pages' absmax / 7, zero point fixed at 8


def quantize(w, K: int, N: int, mode: int = QUANT_ASYM):
    """binary16 W[N, K] (bit patterns) -> (qweight [N, K/8] uint32, scales
    [N, K/128] uint16 (binary16), zeros [N, K/128] uint8), canonical layout."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    if w.shape != (N, K) or K % GROUP or mode not in (QUANT_ASYM, QUANT_SYM):
        raise ValueError("w must be [N, K] with K a multiple of 128, mode 0 or 1")
    qweight = np.empty((N, K // 8), dtype=np.uint32)
    scales = np.empty((N, K // GROUP), dtype=np.uint16)
    zeros = np.empty((N, K // GROUP), dtype=np.uint8)
    _load().w4o_quantize(_ptr(w), K, N, mode, _ptr(qweight), _ptr(scales), _ptr(zeros))
    return qweight, scales, zeros


def gemv_swiglu_f64(qweight, scales, zeros, x, M: int, K: int, I: int):
    """y[M, I] = silu(gate . x) * (up . x) in fp64 for the fused [2I, K] weight
    (gate rows 0..I-1, up rows I..2I-1)."""
    qweight, scales, zeros = _check(qweight, scales, zeros, K, 2 * I)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.shape != (M, K):
        raise ValueError("x must be [M, K]")
    y = np.empty((M, I), dtype=np.float64)
    _load().w4o_gemv_swiglu_f64(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), M, K, I,
                                _ptr(y))
    return y
