"""Thin ctypes binding to libw4.so (include/w4.h).  Argument marshalling only:
every step of the computation runs in the library's CUDA kernels.

Tensors are torch CUDA tensors (torch is used for device memory and streams).
Each function enqueues on the given stream, or on torch's current stream of the
tensor's device when ``stream`` is None, and raises W4Error on a non-OK status.
Importing this module raises if the CUDA library has not been built.
"""
from __future__ import annotations

import ctypes
import enum
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4.so")
HEADER_BYTES = 128
GROUP = 128
MAX_TOKENS = 8
STATIC_SCRATCH_BYTES = 4 * 1024 * 1024   # W4_STATIC_SCRATCH_BYTES

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I = ctypes.c_int
_ST = ctypes.c_int


def _decl(name, res, *args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_status_string = _decl("w4_status_string", ctypes.c_char_p, _ST)
_version = _decl("w4_version", _I)
_repacked_sizes = _decl("w4_repacked_sizes", _ST, _I, _I, ctypes.POINTER(ctypes.c_size_t),
                        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t))
_repack = _decl("w4_repack", _ST, _P, _P, _P, _I, _I, _P, _P, _P, _P)
_check_header = _decl("w4_check_header", _ST, _P, _I, _I)
_dequant = _decl("w4_dequant", _ST, _P, _P, _P, _I, _I, _P, _P)
_gemv = _decl("w4_gemv", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_gemv_f32 = _decl("w4_gemv_f32", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_repacked_sizes_swiglu = _decl("w4_repacked_sizes_swiglu", _ST, _I, _I,
                               ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t),
                               ctypes.POINTER(ctypes.c_size_t))
_repack_swiglu = _decl("w4_repack_swiglu", _ST, _P, _P, _P, _I, _I, _P, _P, _P, _P)
_check_header_swiglu = _decl("w4_check_header_swiglu", _ST, _P, _I, _I)
_gemv_swiglu = _decl("w4_gemv_swiglu", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_gemv_swiglu_f32 = _decl("w4_gemv_swiglu_f32", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_quantize = _decl("w4_quantize", _ST, _P, _I, _I, _I, _P, _P, _P, _P)
_gemv_ws_static = _decl("w4_gemv_ws_static", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_selftest_bounded_wait = _decl("w4_selftest_bounded_wait", _ST, _P, _P)
_stream_read = _decl("w4_stream_read", _ST, _P, ctypes.c_size_t, _I, _P, _P)
_gemm = _decl("w4_gemm", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_gemm_f32 = _decl("w4_gemm_f32", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P)
_gemv_config = _decl("w4_gemv_config", _ST, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I),
                     ctypes.POINTER(_I))


class _LaunchInfo(ctypes.Structure):
    _fields_ = [("k_splits", _I), ("zero_point_folded", _I), ("grid_x", _I), ("grid_y", _I),
                ("persistent", _I), ("overlap", _I), ("capped", _I), ("ring_stages", _I),
                ("wide_prologue", _I), ("blocks_per_sm_max", _I),
                ("smem_bytes", ctypes.c_size_t)]


_gemv_plan = _decl("w4_gemv_plan", _ST, _I, _I, _I, ctypes.POINTER(_LaunchInfo))
_gemv_workspace_bytes = _decl("w4_gemv_workspace_bytes", _ST, _I, _I,
                              ctypes.POINTER(ctypes.c_size_t))
_gemv_ws = _decl("w4_gemv_ws", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P, ctypes.c_size_t, _P)
_gemv_ws_f32 = _decl("w4_gemv_ws_f32", _ST, _P, _P, _P, _P, _P, _I, _I, _I, _P, ctypes.c_size_t,
                     _P)


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    LAYOUT = 3
    CUDA = 4
    SCRATCH_LIMIT = 5


class W4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status: int) -> str:
    return _status_string(int(status)).decode()


def library_path() -> str:
    return LIB_PATH


def version() -> int:
    return _version()


def _ok(status: int, where: str) -> None:
    if status != 0:
        raise W4Error(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream, like: torch.Tensor):
    if stream is None:
        stream = torch.cuda.current_stream(like.device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def repacked_sizes(K: int, N: int):
    """Byte sizes (qweight, scales, zeros) of the kernel layout for N x K."""
    q, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _ok(_repacked_sizes(K, N, ctypes.byref(q), ctypes.byref(s), ctypes.byref(z)),
        "w4_repacked_sizes")
    return q.value, s.value, z.value


def repack(qweight, scales, zeros, K: int, N: int, qweight_out, scales_out, zeros_out,
           stream=None) -> None:
    """w4_repack: canonical device tensors -> the three kernel-layout buffers."""
    _ok(_repack(_ptr(qweight), _ptr(scales), _ptr(zeros), K, N, _ptr(qweight_out),
                _ptr(scales_out), _ptr(zeros_out), _stream(stream, qweight)), "w4_repack")


def check_header(header_bytes: bytes, K: int, N: int) -> None:
    buf = ctypes.create_string_buffer(bytes(header_bytes), HEADER_BYTES)
    _ok(_check_header(ctypes.cast(buf, ctypes.c_void_p), K, N), "w4_check_header")


def dequant(qweight, scales, zeros, K: int, N: int, w_out, stream=None) -> None:
    """w4_dequant: canonical weights -> binary16 [N, K] (bit patterns in w_out)."""
    _ok(_dequant(_ptr(qweight), _ptr(scales), _ptr(zeros), K, N, _ptr(w_out),
                 _stream(stream, qweight)), "w4_dequant")


def gemv(qweight, scales, zeros, x, y, M: int, K: int, N: int, stream=None) -> None:
    """w4_gemv: y[M, N] (bfloat16) = W x with W in the kernel layout."""
    _ok(_gemv(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
              _stream(stream, x)), "w4_gemv")


def gemv_f32(qweight, scales, zeros, x, y, M: int, K: int, N: int, stream=None) -> None:
    """w4_gemv_f32: as gemv but y is float32 (before the bfloat16 cast)."""
    _ok(_gemv_f32(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
                  _stream(stream, x)), "w4_gemv_f32")


def gemm(qweight, scales, zeros, x, y, M: int, K: int, N: int, stream=None) -> None:
    """w4_gemm: y[M, N] (bfloat16) for any M >= 1 (M <= 16: w4_gemv in passes
    of 8; more: one tensor-core pass over the weight)."""
    _ok(_gemm(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
              _stream(stream, x)), "w4_gemm")


def gemm_f32(qweight, scales, zeros, x, y, M: int, K: int, N: int, stream=None) -> None:
    """w4_gemm_f32: as gemm, fp32 result."""
    _ok(_gemm_f32(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
                  _stream(stream, x)), "w4_gemm_f32")


def gemv_workspace_bytes(K: int, N: int) -> int:
    """Bytes of workspace gemv_ws needs for N x K on the current device."""
    n = ctypes.c_size_t()
    _ok(_gemv_workspace_bytes(K, N, ctypes.byref(n)), "w4_gemv_workspace_bytes")
    return n.value


def workspace_counter_bytes(N: int) -> int:
    """Bytes of the row-block counters at the start of a gemv_ws workspace."""
    return ((N + 127) // 128 * 4 + 255) // 256 * 256


def workspace(K: int, N: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor for gemv_ws (allocated by torch)."""
    return torch.zeros(gemv_workspace_bytes(K, N), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def gemv_ws(qweight, scales, zeros, x, y, M: int, K: int, N: int, workspace,
            stream=None) -> None:
    """w4_gemv_ws: as gemv, split evenly over one wave, combining through
    `workspace` (zero-filled before first use; each call leaves its counters,
    the first workspace_counter_bytes(N) bytes, at zero)."""
    _ok(_gemv_ws(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                 _stream(stream, x)), "w4_gemv_ws")


def gemv_ws_f32(qweight, scales, zeros, x, y, M: int, K: int, N: int, workspace,
                stream=None) -> None:
    """w4_gemv_ws_f32: gemv_ws writing the fp32 result."""
    _ok(_gemv_ws_f32(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                     _stream(stream, x)), "w4_gemv_ws_f32")


def gemv_ws_static(qweight, scales, zeros, x, y, M: int, K: int, N: int, stream=None) -> None:
    """w4_gemv_ws_static: gemv_ws with the library's static device scratch
    (allocates nothing).  Calls on one device must not overlap on the GPU;
    the first call on a device should come before any stream capture."""
    _ok(_gemv_ws_static(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, N,
                        _stream(stream, x)), "w4_gemv_ws_static")


def repacked_sizes_swiglu(K: int, I: int):
    """Byte sizes (qweight, scales, zeros) of the gate/up-interleaved layout."""
    q, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _ok(_repacked_sizes_swiglu(K, I, ctypes.byref(q), ctypes.byref(s), ctypes.byref(z)),
        "w4_repacked_sizes_swiglu")
    return q.value, s.value, z.value


def repack_swiglu(qweight, scales, zeros, K: int, I: int, qweight_out, scales_out, zeros_out,
                  stream=None) -> None:
    """w4_repack_swiglu: fused [2I, K] gate/up weight -> interleaved kernel layout."""
    _ok(_repack_swiglu(_ptr(qweight), _ptr(scales), _ptr(zeros), K, I, _ptr(qweight_out),
                       _ptr(scales_out), _ptr(zeros_out), _stream(stream, qweight)),
        "w4_repack_swiglu")


def check_header_swiglu(header_bytes: bytes, K: int, I: int) -> None:
    buf = ctypes.create_string_buffer(bytes(header_bytes), HEADER_BYTES)
    _ok(_check_header_swiglu(ctypes.cast(buf, ctypes.c_void_p), K, I), "w4_check_header_swiglu")


def gemv_swiglu(qweight, scales, zeros, x, y, M: int, K: int, I: int, stream=None) -> None:
    """w4_gemv_swiglu: y[M, I] (bfloat16) = silu(gate x) * (up x)."""
    _ok(_gemv_swiglu(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, I,
                     _stream(stream, x)), "w4_gemv_swiglu")


def gemv_swiglu_f32(qweight, scales, zeros, x, y, M: int, K: int, I: int, stream=None) -> None:
    """w4_gemv_swiglu_f32: the fp32 result."""
    _ok(_gemv_swiglu_f32(_ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(x), _ptr(y), M, K, I,
                         _stream(stream, x)), "w4_gemv_swiglu_f32")


QUANT_ASYMMETRIC = 0      # W4_QUANT_ASYMMETRIC
QUANT_SYMMETRIC = 1       # W4_QUANT_SYMMETRIC


def quantize(w, K: int, N: int, mode: int, qweight, scales, zeros, stream=None) -> None:
    """w4_quantize: binary16 W [N, K] -> canonical qweight, scales, zeros."""
    _ok(_quantize(_ptr(w), K, N, int(mode), _ptr(qweight), _ptr(scales), _ptr(zeros),
                  _stream(stream, w)), "w4_quantize")


def selftest_bounded_wait(status, stream=None) -> None:
    """w4_selftest_bounded_wait: the GEMV kernels' bounded mbarrier wait on a
    barrier nothing completes; `status` (a one-element int32 CUDA tensor)
    becomes 1 when the wait gave up as it must.  About 2 s on the GPU."""
    _ok(_selftest_bounded_wait(_ptr(status), _stream(stream, status)),
        "w4_selftest_bounded_wait")


STREAM_READ_RING = 0      # W4_STREAM_READ_RING
STREAM_READ_LD128 = 1     # W4_STREAM_READ_LD128


def stream_read(src, mode: int, out, stream=None) -> None:
    """w4_stream_read: read all of `src` (a CUDA tensor) once, folding it
    into out[0] (out: two-element int32 CUDA tensor); for measuring the
    read-only bandwidth."""
    _ok(_stream_read(_ptr(src), src.numel() * src.element_size(), int(mode), _ptr(out),
                     _stream(stream, src)), "w4_stream_read")


def gemv_config(K: int, N: int):
    """(16-row tiles per block, K splits, zero point folded) that w4_gemv uses
    for N x K."""
    t, s, f = _I(), _I(), _I()
    _ok(_gemv_config(K, N, ctypes.byref(t), ctypes.byref(s), ctypes.byref(f)), "w4_gemv_config")
    return t.value, s.value, bool(f.value)


def gemv_plan(M: int, K: int, N: int) -> dict:
    """The launch w4_gemv makes for M tokens of an N x K weight on the current
    device (w4_gemv_plan): split, arithmetic, grid, residency, overlap."""
    info = _LaunchInfo()
    _ok(_gemv_plan(M, K, N, ctypes.byref(info)), "w4_gemv_plan")
    return {name: (bool(getattr(info, name)) if name in
                   ("zero_point_folded", "persistent", "overlap", "capped", "wide_prologue")
                   else int(getattr(info, name))) for name, _ in _LaunchInfo._fields_}


@dataclass
class PackedWeight:
    """An N x K weight in the kernel layout (three device buffers)."""
    K: int
    N: int
    qweight: torch.Tensor   # uint8 bytes, starts with the 128-byte header
    scales: torch.Tensor    # uint8 bytes
    zeros: torch.Tensor     # uint8 bytes

    def gemv(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None,
             workspace: torch.Tensor | None = None) -> torch.Tensor:
        """y = W x for x bfloat16 [M, K] on the device; returns y bfloat16 [M, N].
        With a workspace (see `workspace()`), uses gemv_ws."""
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.N), dtype=torch.bfloat16, device=x.device)
        if workspace is None:
            gemv(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.N, stream)
        else:
            gemv_ws(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.N, workspace,
                    stream)
        return y

    def gemv_f32(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None,
                 workspace: torch.Tensor | None = None):
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.N), dtype=torch.float32, device=x.device)
        if workspace is None:
            gemv_f32(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.N, stream)
        else:
            gemv_ws_f32(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.N,
                        workspace, stream)
        return y


def pack(qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, K: int, N: int,
         stream=None) -> PackedWeight:
    """Allocate the kernel-layout buffers (torch), repack into them and check
    the header once."""
    dev = qweight.device
    qb, sb, zb = repacked_sizes(K, N)
    qo = torch.empty(qb, dtype=torch.uint8, device=dev)
    so = torch.empty(sb, dtype=torch.uint8, device=dev)
    zo = torch.empty(zb, dtype=torch.uint8, device=dev)
    repack(qweight, scales, zeros, K, N, qo, so, zo, stream)
    check_header(qo[:HEADER_BYTES].cpu().numpy().tobytes(), K, N)
    return PackedWeight(K, N, qo, so, zo)


@dataclass
class PackedSwiGLU:
    """A fused [2I, K] gate/up weight in the interleaved kernel layout."""
    K: int
    I: int
    qweight: torch.Tensor
    scales: torch.Tensor
    zeros: torch.Tensor

    def gemv(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """y[M, I] = silu(gate x) * (up x), bfloat16."""
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.I), dtype=torch.bfloat16, device=x.device)
        gemv_swiglu(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.I, stream)
        return y

    def gemv_f32(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.I), dtype=torch.float32, device=x.device)
        gemv_swiglu_f32(self.qweight, self.scales, self.zeros, x, y, M, self.K, self.I, stream)
        return y


def pack_swiglu(qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, K: int,
                I: int, stream=None) -> PackedSwiGLU:
    """Allocate the interleaved-layout buffers (torch), repack the fused
    [2I, K] gate/up weight into them and check the header once."""
    dev = qweight.device
    qb, sb, zb = repacked_sizes_swiglu(K, I)
    qo = torch.empty(qb, dtype=torch.uint8, device=dev)
    so = torch.empty(sb, dtype=torch.uint8, device=dev)
    zo = torch.empty(zb, dtype=torch.uint8, device=dev)
    repack_swiglu(qweight, scales, zeros, K, I, qo, so, zo, stream)
    check_header_swiglu(qo[:HEADER_BYTES].cpu().numpy().tobytes(), K, I)
    return PackedSwiGLU(K, I, qo, so, zo)
