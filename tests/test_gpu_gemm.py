"""w4_gemm (any M, passes of 8 tokens) through the C ABI: parity with the
oracle, every row bit-identical to w4_gemv on that token alone, graph capture
and argument errors."""
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


def setup(w4, name, K, N, M, seed):
    p = syn.make_problem(name, K, N, M, seed=seed)
    qw, sc, zp, x = tu.to_device(p)
    return p, w4.pack(qw, sc, zp, K, N), x


@pytest.mark.parametrize("M,K,N", [(9, 896, 1000), (16, 3584, 4608), (33, 256, 200),
                                   (64, 3584, 3584), (17, 18944, 300)])
def test_gemm_parity(w4, M, K, N):
    p, packed, x = setup(w4, f"gemm.{M}.{K}.{N}", K, N, M, 1)
    y32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, y32, M, K, N)
    w4.gemm(packed.qweight, packed.scales, packed.zeros, x, y16, M, K, N)
    torch.cuda.synchronize()
    ref, refabs = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, with_abs=True)
    _, S, fold = w4.gemv_config(K, N)
    mag = tu.folded_abs(p) if fold else refabs
    tu.check_gemv(y32.cpu().numpy(), tu.bf16_bits(y16), ref, mag, K, S, f"gemm M={M}",
                  tu.FOLD_EXTRA_STEPS if fold else 0)


def test_gemm_multi_wave_rows_equal_single_token_gemv(w4):
    """A product of several waves without a K split: passes of 8 and of 4
    tokens run the persistent grid, the single-token products one block per
    row block; every row is the same bit for bit."""
    M, K, N = 20, 1024, 64037
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert w4.gemv_config(K, N)[1] == 1 and (N + 127) // 128 > 3 * sms
    p, packed, x = setup(w4, "gemm.multiwave", K, N, M, 3)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, y, M, K, N)
    for r in (0, 9, 16, 19):
        one = packed.gemv_f32(x[r:r + 1].contiguous())
        assert torch.equal(one[0], y[r]), r


def test_gemm_rows_equal_single_token_gemv(w4):
    M, K, N = 40, 3584, 37888
    p, packed, x = setup(w4, "gemm.rows", K, N, M, 2)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, y, M, K, N)
    for r in (0, 7, 8, 23, 39):
        one = packed.gemv_f32(x[r:r + 1].contiguous())
        assert torch.equal(one[0], y[r]), r
    for m in range(1, 9):                      # M <= 8 is exactly w4_gemv
        a = torch.empty((m, N), dtype=torch.float32, device="cuda")
        w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x[:m].contiguous(), a, m, K, N)
        assert torch.equal(a, packed.gemv_f32(x[:m].contiguous()))


def test_gemm_graph_and_errors(w4):
    M, K, N = 20, 1024, 512
    _, packed, x = setup(w4, "gemm.graph", K, N, M, 3)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    eager = torch.empty_like(y)
    w4.gemm(packed.qweight, packed.scales, packed.zeros, x, eager, M, K, N)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.gemm(packed.qweight, packed.scales, packed.zeros, x, y, M, K, N, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.gemm(packed.qweight, packed.scales, packed.zeros, x, y, M, K, N)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, eager)
    with pytest.raises(w4.W4Error) as e:
        w4.gemm(packed.qweight, packed.scales, packed.zeros, x, y, 0, K, N)
    assert e.value.status == w4.Status.UNSUPPORTED
