"""GPU parity of the fused gate/up product with SwiGLU (w4_repack_swiglu +
w4_gemv_swiglu, through the C ABI) against the oracle's w4o_gemv_swiglu_f64.

Tolerance: relative L2 <= 1e-3 and max |error| <= 1e-2 max |y| on the fp32
output; the bfloat16 output within 1 ulp of RNE(y_ref) except where the fp32
error is within the propagated bound: gate and up carry the fp32
accumulation bounds Bg, Bu of the matrix-vector product (w4_testutil, for
the arithmetic the launch shape uses), silu has slope at most 1.1, and the
fp32 activation and product add a few ulps:
  |y~ - y| <= 1.1 Bg (|u| + Bu) + (|silu(g)| + 1.1 Bg) Bu + 8 * 2^-24 |y|."""
import numpy as np
import pytest

import oracle
from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


def run(w4, p, I, packed=None):
    qw, sc, zp, x = tu.to_device(p)
    if packed is None:
        packed = w4.pack_swiglu(qw, sc, zp, p.K, I)
    y32 = packed.gemv_f32(x)
    y16 = packed.gemv(x)
    torch.cuda.synchronize()
    return y32.cpu().numpy(), tu.bf16_bits(y16), packed


def bound(w4, p, I, cols):
    """Per output (M, len(cols)): the propagated fp32 bound, and the oracle's y."""
    K = p.K
    rows = np.concatenate([cols, I + cols])
    ref, refabs = oracle.gemv_rows_f64(p.qweight, p.scales, p.zeros, p.x, p.M, K, 2 * I, rows,
                                       with_abs=True)
    _, S, fold = w4.gemv_config(K, 16 * ((I + 7) // 8))
    n = 8 + K // 128 + S + 1 + (tu.FOLD_EXTRA_STEPS if fold else 0)
    mag = tu.folded_abs(p, rows) if fold else refabs
    B = n * 2.0 ** -23 * mag
    g, u = ref[:, :len(cols)], ref[:, len(cols):]
    Bg, Bu = B[:, :len(cols)], B[:, len(cols):]
    silu = g / (1.0 + np.exp(-g))
    y = silu * u
    return y, 1.1 * Bg * (np.abs(u) + Bu) + (np.abs(silu) + 1.1 * Bg) * Bu + 8 * 2.0 ** -24 * np.abs(y)


def check(got32, got16, y, b, what):
    err = got32.astype(np.float64) - y
    assert np.linalg.norm(err) <= tu.REL_L2 * np.linalg.norm(y), what
    assert np.abs(err).max() <= tu.MAX_ABS_FRAC * np.abs(y).max(), what
    want16 = oracle.bf16_rne(y.astype(np.float32))
    off = np.abs(tu.ordered(got16) - tu.ordered(want16)) > 1
    assert (np.abs(err[off]) <= b[off]).all(), f"{what}: {int(off.sum())} outputs beyond 1 ulp"
    assert np.array_equal(got16, oracle.bf16_rne(got32)), what


CASES = [(1, 3584, 18944), (8, 3584, 18944), (1, 896, 4864), (2, 5120, 8704), (3, 256, 17),
         (5, 1024, 100), (4, 18944, 24), (1, 128, 1)]


@pytest.mark.parametrize("M,K,I", CASES)
def test_swiglu_parity(w4, M, K, I):
    p = syn.make_problem(f"swiglu.{K}.{I}", K, 2 * I, M, seed=3)
    got32, got16, _ = run(w4, p, I)
    cols = np.arange(I) if I * K * M <= 2 ** 28 else np.unique(np.concatenate(
        [np.arange(64), np.arange(I - 64, I),
         np.random.default_rng(4).choice(I, 1024, replace=False)]))
    y, b = bound(w4, p, I, cols)
    # the oracle's own fused product agrees with the composition used here
    if I * K * M <= 2 ** 26:
        assert np.allclose(oracle.gemv_swiglu_f64(p.qweight, p.scales, p.zeros, p.x, M, K, I),
                           y, rtol=1e-12, atol=0)
    check(got32[:, cols], got16[:, cols], y, b, f"M={M} K={K} I={I}")


def test_swiglu_persistent_grid(w4):
    """Enough rows for several waves without a K split, from three tokens on:
    the persistent grid stores the activation row block by row block."""
    M, K, I = 4, 1024, 30001
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, S, fold = w4.gemv_config(K, 16 * ((I + 7) // 8))
    rows = 16 * ((I + 7) // 8)                 # kernel rows of the interleaved layout
    assert S == 1 and fold and (rows + 127) // 128 > 3 * sms
    p = syn.make_problem(f"swiglu.persist.{K}.{I}", K, 2 * I, M, seed=7)
    got32, got16, _ = run(w4, p, I)
    cols = np.unique(np.concatenate([np.arange(64), np.arange(I - 64, I),
                                     np.random.default_rng(8).choice(I, 1024, replace=False)]))
    y, b = bound(w4, p, I, cols)
    check(got32[:, cols], got16[:, cols], y, b, f"persistent M={M} K={K} I={I}")


def test_swiglu_matches_plain_gemv_then_activation(w4):
    """The interleaved layout only reorders rows: the gate and up products
    are the plain w4_gemv_f32 results (same split, same arithmetic)."""
    M, K, I = 2, 3584, 4608
    p = syn.make_problem("swiglu.plain", K, 2 * I, M, seed=5)
    got32, _, _ = run(w4, p, I)
    qw, sc, zp, x = tu.to_device(p)
    plain = w4.pack(qw, sc, zp, K, 2 * I).gemv_f32(x).cpu().numpy().astype(np.float64)
    g, u = plain[:, :I], plain[:, I:]
    want = g / (1.0 + np.exp(-g)) * u
    assert np.abs(got32 - want).max() <= 1e-5 * np.abs(want).max()


def test_swiglu_determinism_batch_invariance_and_graph(w4):
    M, K, I = 8, 3584, 18944
    p = syn.make_problem("swiglu.det", K, 2 * I, M, seed=6)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack_swiglu(qw, sc, zp, K, I)
    first = packed.gemv_f32(x).cpu()
    for _ in range(10):
        assert torch.equal(packed.gemv_f32(x).cpu(), first)
    for r in (0, 5):
        assert torch.equal(packed.gemv_f32(x[r:r + 1].contiguous()).cpu()[0], first[r])
    y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    eager = packed.gemv(x).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        packed.gemv(x, y, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        packed.gemv(x, y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, eager)


def test_swiglu_header_and_errors(w4):
    K, I = 256, 40
    p = syn.make_problem("swiglu.hdr", K, 2 * I, 2, seed=7)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack_swiglu(qw, sc, zp, K, I)
    hdr = packed.qweight[:128].cpu().numpy().tobytes()
    w4.check_header_swiglu(hdr, K, I)
    with pytest.raises(w4.W4Error):
        w4.check_header(hdr, K, I)                 # not the plain layout
    with pytest.raises(w4.W4Error):
        w4.check_header_swiglu(hdr, K, I + 8)
    y = torch.empty((9, I), dtype=torch.bfloat16, device="cuda")
    x9 = torch.zeros((9, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.gemv_swiglu(packed.qweight, packed.scales, packed.zeros, x9, y, 9, K, I)
    assert e.value.status == w4.Status.UNSUPPORTED
    with pytest.raises(w4.W4Error) as e:
        w4.gemv_swiglu(packed.qweight, packed.scales, packed.zeros, x, y, 2, 200, I)
    assert e.value.status == w4.Status.INVALID_ARG
