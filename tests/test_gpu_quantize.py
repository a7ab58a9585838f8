"""GPU parity of w4_quantize (through the C ABI) against the oracle's
quantiser: the codes, scales and zero points are integers or bit patterns,
so they must be identical.  Both sides take every decision in fp32 with
correctly rounded operations (the oracle in C, the kernel with the
round-to-nearest intrinsics)."""
import numpy as np
import pytest

import oracle
from tests import test_oracle_quantize as qpins

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


def gpu_quantize(w4, w16: np.ndarray, mode: int):
    N, K = w16.shape
    wd = torch.from_numpy(np.ascontiguousarray(w16).view(np.int16)).cuda()
    qw = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((N, K // 128), dtype=torch.int16, device="cuda")
    zp = torch.empty((N, K // 128), dtype=torch.uint8, device="cuda")
    w4.quantize(wd, K, N, mode, qw, sc, zp)
    torch.cuda.synchronize()
    return (qw.cpu().numpy().view(np.uint32), sc.cpu().numpy().view(np.uint16),
            zp.cpu().numpy())


def weights(N, K, seed):
    """fp16 weights with row magnitudes from 2^-20 to 2^6 and a few special
    rows: all zero, constant, subnormal only, the fp16 extremes, half-integers
    (ties for the rounding)."""
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-20, 6, size=(N, 1)))
    w = (rng.standard_normal((N, K)) * mag).astype(np.float16)
    if N >= 6:
        w[0] = 0
        w[1] = np.float16(-0.375)
        w[2] = (rng.integers(-40, 40, size=K) * 2.0 ** -24).astype(np.float16)   # subnormals
        w[3, ::2], w[3, 1::2] = np.float16(65504), np.float16(-65504)
        w[4] = (rng.integers(-16, 16, size=K) / 2.0).astype(np.float16)
        w[5, : K // 2] = -0.0
    assert np.isfinite(w).all()
    return w


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 1152), (1000, 896), (3584, 3584),
                                 (37888, 3584)])
def test_quantize_bit_exact(w4, mode, N, K):
    w = weights(N, K, seed=N + K + mode)
    got = gpu_quantize(w4, w, mode)
    want = oracle.quantize(w.view(np.uint16), K, N, mode)
    for g, o, name in zip(got, want, ("qweight", "scales", "zeros")):
        assert np.array_equal(g, o), f"{name} differs at {np.argwhere(g != o)[:5]}"


@pytest.mark.parametrize("case", qpins._groups(), ids=lambda c: c[0])
def test_quantize_golden_groups(w4, case):
    gid, mode, period, vals, scale, zero, qs = case
    K = 256
    w = np.array([[vals[k % period] for k in range(K)]], np.float16)
    qw, sc, zp = gpu_quantize(w4, w, mode)
    assert list(sc[0]) == [scale, scale] and list(zp[0]) == [zero, zero]
    assert list(qpins._nibbles(qw, K)[0]) == [qs[k % period] for k in range(K)]


def test_quantize_then_gemv(w4):
    """The quantiser's output feeds the product unchanged (canonical layout):
    quantise on the GPU, pack, multiply, and compare with the oracle's product
    of the oracle's quantisation."""
    from int4_weight_only_w4_gb300 import synthetic as syn
    from tests import w4_testutil as tu
    N, K, M = 512, 2048, 3
    w = weights(N, K, seed=77)
    qw, sc, zp = gpu_quantize(w4, w, 0)
    x = syn.make_x("quant.x", M, K, 0)
    p = syn.Problem("quant", M, K, N, qw, sc, zp, x)
    qd, sd, zd, xd = tu.to_device(p)
    packed = w4.pack(qd, sd, zd, K, N)
    y32 = packed.gemv_f32(xd).cpu().numpy()
    ref = oracle.gemv_f64(*oracle.quantize(w.view(np.uint16), K, N, 0), x, M, K, N)
    assert np.linalg.norm(y32 - ref) <= 1e-3 * np.linalg.norm(ref)


def test_quantize_argument_errors(w4):
    K, N = 256, 4
    w = torch.zeros((N, K), dtype=torch.int16, device="cuda")
    qw = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((N, 2), dtype=torch.int16, device="cuda")
    zp = torch.empty((N, 2), dtype=torch.uint8, device="cuda")
    for bad in [dict(mode=2), dict(K=200)]:
        args = dict(K=K, N=N, mode=0)
        args.update(bad)
        with pytest.raises(w4.W4Error) as e:
            w4.quantize(w, args["K"], args["N"], args["mode"], qw, sc, zp)
        assert e.value.status == w4.Status.INVALID_ARG
    # weights that start 2 bytes past a 16-byte boundary
    buf = torch.zeros(N * K + 8, dtype=torch.int16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.quantize(buf[1:1 + N * K], K, N, 0, qw, sc, zp)
    assert e.value.status == w4.Status.INVALID_ARG


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_outputs_at_minimum_alignment(w4, mode):
    """qweight need only be 4-byte aligned, scales 2-byte aligned and zeros
    not aligned at all: outputs written one element past aligned buffers
    equal the aligned call's."""
    N, K = 65, 1152
    w = weights(N, K, seed=77 + mode)
    want = gpu_quantize(w4, w, mode)
    wd = torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).cuda()
    qw = torch.empty(N * K // 8 + 1, dtype=torch.int32, device="cuda")
    sc = torch.empty(N * K // 128 + 1, dtype=torch.int16, device="cuda")
    zp = torch.empty(N * K // 128 + 1, dtype=torch.uint8, device="cuda")
    assert qw[1:].data_ptr() % 8 == 4
    w4.quantize(wd, K, N, mode, qw[1:], sc[1:], zp[1:])
    torch.cuda.synchronize()
    got = (qw[1:].cpu().numpy().view(np.uint32).reshape(N, K // 8),
           sc[1:].cpu().numpy().view(np.uint16).reshape(N, K // 128),
           zp[1:].cpu().numpy().reshape(N, K // 128))
    for g, o, name in zip(got, want, ("qweight", "scales", "zeros")):
        assert np.array_equal(g, o), name

