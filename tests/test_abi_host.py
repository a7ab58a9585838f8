"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/w4.h declares, and rejects bad arguments before it
touches the device.  Every call here fails argument validation, so no pointer
is ever dereferenced and no kernel is launched."""
import ctypes
import os
import re
import struct

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4.h")
LIB = os.path.join(ROOT, "int4_weight_only_w4_gb300", "libw4.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"libw4.so does not export {n}"


def test_binding_names_match_abi():
    from int4_weight_only_w4_gb300 import w4
    for n in declared_functions():
        assert hasattr(w4, n[len("w4_"):]), n


def test_status_strings(lib):
    lib.w4_status_string.restype = ctypes.c_char_p
    for code, name in enumerate(["W4_OK", "W4_ERR_INVALID_ARG", "W4_ERR_UNSUPPORTED",
                                 "W4_ERR_LAYOUT", "W4_ERR_CUDA", "W4_ERR_SCRATCH_LIMIT"]):
        assert lib.w4_status_string(code).decode() == name
    assert lib.w4_status_string(99).decode() == "W4_ERR_UNKNOWN"


def sizes(lib, K, N):
    q, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    st = lib.w4_repacked_sizes(K, N, ctypes.byref(q), ctypes.byref(s), ctypes.byref(z))
    return st, q.value, s.value, z.value


@pytest.mark.parametrize("K,N", [(128, 1), (3584, 37888), (18944, 3584), (256, 17)])
def test_repacked_sizes(lib, K, N):
    st, q, s, z = sizes(lib, K, N)
    blocks = (N + 127) // 128
    assert st == 0
    assert q == 128 + blocks * (K // 128) * 8192
    assert s == blocks * (K // 128) * 256
    assert z == blocks * (K // 128) * 64


@pytest.mark.parametrize("K,N", [(0, 8), (100, 8), (128, 0), (-128, 4)])
def test_repacked_sizes_rejects(lib, K, N):
    assert sizes(lib, K, N)[0] == 1


P = ctypes.c_void_p
FAKE = 0x10000          # 16-byte aligned, never dereferenced (validation fails first)


def gemv(lib, q=FAKE, s=FAKE, z=FAKE, x=FAKE, y=FAKE, M=1, K=128, N=16):
    lib.w4_gemv.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    return lib.w4_gemv(q, s, z, x, y, M, K, N, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), 1), (dict(s=None), 1), (dict(z=None), 1), (dict(x=None), 1),
    (dict(y=None), 1), (dict(K=100), 1), (dict(K=0), 1), (dict(N=0), 1),
    (dict(M=0), 2), (dict(M=9), 2), (dict(q=FAKE + 8), 1), (dict(s=FAKE + 4), 1),
    (dict(z=FAKE + 8), 1), (dict(x=FAKE + 8), 1), (dict(y=FAKE + 1), 1),
])
def test_gemv_argument_errors(lib, kw, want):
    assert gemv(lib, **kw) == want


def gemm(lib, q=FAKE, s=FAKE, z=FAKE, x=FAKE, y=FAKE, M=17, K=128, N=16):
    lib.w4_gemm.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    return lib.w4_gemm(q, s, z, x, y, M, K, N, None)


# w4_gemm above 16 tokens (the tensor-core path): every case fails validation
# before the device is touched.  1 = W4_ERR_INVALID_ARG, 2 = W4_ERR_UNSUPPORTED.
@pytest.mark.parametrize("kw,want", [
    (dict(M=0), 2), (dict(M=-3), 2), (dict(K=100), 1), (dict(N=0), 1),
    (dict(q=None), 1), (dict(s=None), 1), (dict(z=None), 1), (dict(x=None), 1),
    (dict(y=None), 1), (dict(q=FAKE + 8), 1), (dict(s=FAKE + 4), 1), (dict(z=FAKE + 8), 1),
    (dict(x=FAKE + 8), 1), (dict(y=FAKE + 1), 1),
    # more than 65535 tiles of 128 tokens
    (dict(M=65536 * 128 + 1, K=128), 2),
    # M * K >= 2^40
    (dict(M=1 << 22, K=1 << 18), 2),
    # a weight of 2^25 or more 128 x 128 records (tensor-copy rows past 2^31)
    (dict(M=17, K=128 * 1024, N=32768 * 128), 2),
])
def test_gemm_argument_errors(lib, kw, want):
    assert gemm(lib, **kw) == want


def test_gemv_ws_argument_errors(lib):
    lib.w4_gemv_ws.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                               ctypes.c_size_t, P]
    assert lib.w4_gemv_ws(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 16, None, 1 << 20, None) == 1
    assert lib.w4_gemv_ws(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 16, FAKE + 16, 1 << 20,
                          None) == 1
    assert lib.w4_gemv_ws(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 128, 16, FAKE, 1 << 20, None) == 2
    lib.w4_gemv_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, P]
    assert lib.w4_gemv_workspace_bytes(100, 16, FAKE) == 1


def test_dequant_and_repack_argument_errors(lib):
    lib.w4_dequant.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, P]
    assert lib.w4_dequant(None, FAKE, FAKE, 128, 4, FAKE, None) == 1
    assert lib.w4_dequant(FAKE + 4, FAKE, FAKE, 128, 4, FAKE, None) == 1
    assert lib.w4_dequant(FAKE, FAKE, FAKE, 130, 4, FAKE, None) == 1
    lib.w4_repack.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P]
    assert lib.w4_repack(FAKE, FAKE, FAKE, 128, 4, None, FAKE, FAKE, None) == 1
    assert lib.w4_repack(FAKE, FAKE, FAKE, 128, 4, FAKE + 4, FAKE, FAKE, None) == 1
    assert lib.w4_repack(FAKE, FAKE, FAKE, 64, 4, FAKE, FAKE, FAKE, None) == 1


def header(K, N, magic=b"W4G128KL", layout=1, version=4, bad=0, kerr=0):
    return magic + struct.pack("<IIiiII", layout, version, K, N, bad, kerr) + bytes(96)


@pytest.mark.parametrize("mut,want", [
    (dict(), 0), (dict(magic=b"W4G128XX"), 3), (dict(layout=2), 3), (dict(version=9), 3),
    (dict(K=256), 3), (dict(N=17), 3), (dict(bad=1), 3), (dict(kerr=1), 4),
])
def test_check_header(lib, mut, want):
    args = dict(K=384, N=64)
    args.update(mut)
    buf = ctypes.create_string_buffer(header(**args), 128)
    lib.w4_check_header.argtypes = [P, ctypes.c_int, ctypes.c_int]
    assert lib.w4_check_header(ctypes.cast(buf, P), 384, 64) == want
    assert lib.w4_check_header(None, 384, 64) == 1


def test_selftest_argument_errors(lib):
    lib.w4_selftest_bounded_wait.restype = ctypes.c_int
    lib.w4_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert lib.w4_selftest_bounded_wait(None, None) == 1           # INVALID_ARG
    assert lib.w4_selftest_bounded_wait(0x1002, None) == 1         # not 4-byte aligned

