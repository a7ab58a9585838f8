"""w4_gemm (any M) through the C ABI.  Up to 16 tokens it is w4_gemv in
passes of 8 (each row the single-token product, bit for bit); more tokens run
the single-pass tensor-core kernel (tiles of up to 128 tokens, one pass over
the weight).  Parity with the oracle over several tiles, ragged tiles, a
single group, K splits and the full-size 7B gate_up, down and LM head
(sampled rows); a token's result independent of M and of the other tokens;
repeatability; graph capture and argument errors."""
import numpy as np
import pytest

import oracle
from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# The tensor-core kernel splits K over at most 8 blocks of a cluster: the
# bound's split term uses that maximum.
TC_MAX_SPLITS = 8


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


def setup(w4, name, K, N, M, seed):
    p = syn.make_problem(name, K, N, M, seed=seed)
    qw, sc, zp, x = tu.to_device(p)
    return p, w4.pack(qw, sc, zp, K, N), x


def run(w4, packed, x, M, K, N):
    y32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, y32, M, K, N)
    w4.gemm(packed.qweight, packed.scales, packed.zeros, x, y16, M, K, N)
    torch.cuda.synchronize()
    return y32, y16


def sample_rows(N, rng, count=1536):
    if N <= count:
        return np.arange(N)
    mid = rng.choice(np.arange(64, N - 64), size=count - 128, replace=False)
    return np.sort(np.concatenate([np.arange(64), mid, np.arange(N - 64, N)]))


# (M, K, N): one and several 128-token tiles with ragged last tiles; one group
# (K = 128); row counts that are not a multiple of 128; shapes whose K is
# split over a cluster (few row blocks, long K) and shapes that take more than
# one wave of blocks (many row blocks).
TC_CASES = [(17, 896, 1000), (24, 3584, 4608), (17, 18944, 300), (33, 256, 200),
            (64, 3584, 3584), (128, 896, 1152), (129, 1024, 640), (200, 4864, 896),
            (300, 128, 256), (40, 1152, 40000),
            # one output row; a few rows under a K split of 8; one group and a
            # ragged second tile; a tile of exactly 16 tokens past the first
            (20, 128, 1), (70, 18944, 40), (150, 128, 130), (144, 2048, 2000)]


@pytest.mark.parametrize("M,K,N", TC_CASES)
def test_gemm_tc_parity(w4, M, K, N):
    p, packed, x = setup(w4, f"gemm.{M}.{K}.{N}", K, N, M, 1)
    y32, y16 = run(w4, packed, x, M, K, N)
    rows = sample_rows(N, np.random.default_rng(7)) if M * N * K > 2 ** 30 else np.arange(N)
    ref, refabs = oracle.gemv_rows_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, rows,
                                       with_abs=True)
    tu.check_gemv(y32.cpu().numpy()[:, rows], tu.bf16_bits(y16)[:, rows], ref, refabs, K,
                  TC_MAX_SPLITS, f"gemm M={M} K={K} N={N}")


@pytest.mark.parametrize("name,M", [("qwen7b.gate_up", 128), ("qwen7b.down", 96),
                                    ("qwen7b.lm_head", 64)])
def test_gemm_tc_full_size_sampled(w4, name, M):
    """Full-size 7B products (the shapes `bench.py --gemm` times), compared with
    the oracle on a sample of rows that includes the first and last row blocks."""
    _, K, N, _, srange = syn.shape(name)
    p = syn.make_problem(f"{name}.gemm.M{M}", K, N, M, seed=4, scale_range=srange)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack(qw, sc, zp, K, N)
    y32, y16 = run(w4, packed, x, M, K, N)
    rows = sample_rows(N, np.random.default_rng(11), 1024)
    ref, refabs = oracle.gemv_rows_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, rows,
                                       with_abs=True)
    tu.check_gemv(y32.cpu().numpy()[:, rows], tu.bf16_bits(y16)[:, rows], ref, refabs, K,
                  TC_MAX_SPLITS, f"{name} gemm M={M}")


@pytest.mark.parametrize("K,N", [(3584, 4608), (18944, 896), (1024, 37888)])
def test_gemm_tc_token_independent_of_batch(w4, K, N):
    """A token's fp32 result is the same bit for bit whatever M is and
    whichever tokens share its tile (the K split depends on K, N and the SM
    count only; every token column is summed on its own)."""
    M = 140
    p, packed, x = setup(w4, f"gemm.inv.{K}.{N}", K, N, M, 5)
    full = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, full, M, K, N)
    for lo, hi in ((0, 17), (0, 128), (120, 140), (5, 30), (100, 140)):
        m = hi - lo
        part = torch.empty((m, N), dtype=torch.float32, device="cuda")
        w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x[lo:hi].contiguous(), part, m,
                    K, N)
        torch.cuda.synchronize()
        assert torch.equal(part, full[lo:hi]), (lo, hi)


def test_gemm_tc_repeatable(w4):
    M, K, N = 77, 18944, 3584
    p, packed, x = setup(w4, "gemm.rep", K, N, M, 6)
    first = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, first, M, K, N)
    again = torch.empty_like(first)
    for _ in range(20):
        w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, again, M, K, N)
        torch.cuda.synchronize()
        assert torch.equal(again, first)
    w4.check_header(packed.qweight[:128].cpu().numpy().tobytes(), K, N)   # no kernel error


def test_gemm_up_to_16_tokens_is_gemv_in_passes(w4):
    M, K, N = 16, 3584, 37888
    p, packed, x = setup(w4, "gemm.le16", K, N, M, 2)
    for m in range(1, 17):
        a = torch.empty((m, N), dtype=torch.float32, device="cuda")
        w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x[:m].contiguous(), a, m, K, N)
        # pass 1: tokens 0..7, pass 2: tokens 8..m-1, each exactly w4_gemv
        assert torch.equal(a[:8], packed.gemv_f32(x[:min(m, 8)].contiguous()))
        if m > 8:
            assert torch.equal(a[8:], packed.gemv_f32(x[8:m].contiguous()))
    # and each row is the single-token product
    a = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, a, M, K, N)
    for r in (0, 7, 8, 15):
        assert torch.equal(a[r], packed.gemv_f32(x[r:r + 1].contiguous())[0]), r


def test_gemm_no_write_outside_y(w4):
    """The tensor-core kernel writes y[M][N] and nothing around it."""
    M, K, N = 37, 1024, 300
    p, packed, x = setup(w4, "gemm.guard", K, N, M, 8)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    w4.gemm_f32(packed.qweight, packed.scales, packed.zeros, x, y, M, K, N)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == -7.0).all()) and bool((buf[pad + M * N:] == -7.0).all())
    ref = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N)
    assert np.abs(y.cpu().numpy() - ref).max() <= 1e-4 * np.abs(ref).max()


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
    # x must be 16-byte aligned for the tensor copies
    xs = torch.empty(M * K + 8, dtype=torch.bfloat16, device="cuda")[1:1 + M * K].view(M, K)
    with pytest.raises(w4.W4Error) as e:
        w4.gemm(packed.qweight, packed.scales, packed.zeros, xs, y, M, K, N)
    assert e.value.status == w4.Status.INVALID_ARG
