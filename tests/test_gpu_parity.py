"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Dequantisation must be bit-exact; the GEMV must meet the
tolerances in w4_testutil.  Closed-form cases are exact where the arithmetic
makes them so (one-hot x and power-of-two scaling on both splits; q = z and the
identity pattern on the workspace split, whose tensor-core operand is q - z
exactly) and within the derived fp32 bound otherwise (the cluster split folds
the zero point out of the inner product)."""
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


PATHS = ["cluster", "ws"]     # w4_gemv (cluster split) and w4_gemv_ws (workspace split)


def run_gemv(w4, p, packed=None, path="cluster"):
    qw, sc, zp, x = tu.to_device(p)
    if packed is None:
        packed = w4.pack(qw, sc, zp, p.K, p.N)
    ws = w4.workspace(p.K, p.N) if path == "ws" else None
    y32 = packed.gemv_f32(x, workspace=ws)
    y16 = packed.gemv(x, workspace=ws)
    torch.cuda.synchronize()
    if ws is not None:
        counters = ws[:w4.workspace_counter_bytes(p.N)]
        assert int(counters.count_nonzero()) == 0, "workspace counters not left at zero"
    return y32.cpu().numpy(), tu.bf16_bits(y16), packed


def path_splits(w4, path, K, N):
    """Upper bound on the partial sums combined per output: the cluster split
    uses gemv_config's count; the workspace split cuts a row at group
    boundaries, so at most one piece per group."""
    return w4.gemv_config(K, N)[1] if path == "cluster" else K // 128


def folds(w4, path, K, N):
    """Whether the path folds the zero point out of the inner product."""
    return path == "cluster" and w4.gemv_config(K, N)[2]


def bound_terms(w4, path, p, rows, refabs):
    """(magnitudes, extra rounding steps) of the fp32 bound for a path."""
    if folds(w4, path, p.K, p.N):
        return tu.folded_abs(p, rows), tu.FOLD_EXTRA_STEPS
    return refabs, 0


def oracle_rows(p, rows):
    return oracle.gemv_rows_f64(p.qweight, p.scales, p.zeros, p.x, p.M, p.K, p.N, rows,
                                with_abs=True)


def sample_rows(N, rng, count=1536):
    if N <= count:
        return np.arange(N)
    head = np.arange(64)
    tail = np.arange(N - 64, N)
    mid = rng.choice(np.arange(64, N - 64), size=count - 128, replace=False)
    return np.sort(np.concatenate([head, mid, tail]))


# ---- dequantisation: bit-exact -------------------------------------------------

@pytest.mark.parametrize("name", [s[0] for s in syn.SHAPES])
def test_dequant_bit_exact(w4, name):
    _, K, N, _, srange = syn.shape(name)
    qwn, scn, zpn = syn.make_weights(name, K, N, seed=0, scale_range=srange)
    p = syn.Problem(name, 1, K, N, qwn, scn, zpn, np.zeros((1, K), np.uint16))
    qw, sc, zp, _ = tu.to_device(p)
    out = torch.empty((N, K), dtype=torch.int16, device="cuda")
    w4.dequant(qw, sc, zp, K, N, out)
    got = out.cpu().numpy().view(np.uint16)
    if N * K > 64 * 2 ** 20:      # compare a row sample on the largest weights
        rows = sample_rows(N, np.random.default_rng(0), 2048)
        want = oracle.dequant_f16(qwn[rows], scn[rows], zpn[rows], K, len(rows))
        assert np.array_equal(got[rows], want)
    else:
        assert np.array_equal(got, oracle.dequant_f16(qwn, scn, zpn, K, N))


def test_dequant_extreme_scales(w4):
    rng = np.random.default_rng(3)
    K, N = 256, 40
    q = syn.uniform_words(1, "dq", (N, K // 8))
    sc = rng.choice(np.array([0x0001, 0x03FF, 0x0400, 0x7BFF, 0x5A00, 0x3C01, 0x8001, 0xBC00],
                             np.uint16), size=(N, 2))
    zp = rng.integers(0, 16, size=(N, 2)).astype(np.uint8)
    p = syn.Problem("dq", 1, K, N, q, sc, zp, np.zeros((1, K), np.uint16))
    qw, scd, zpd, _ = tu.to_device(p)
    out = torch.empty((N, K), dtype=torch.int16, device="cuda")
    w4.dequant(qw, scd, zpd, K, N, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), oracle.dequant_f16(q, sc, zp, K, N))


# ---- GEMV at the workload shapes ------------------------------------------------

CASES = [(name, M) for (name, K, N, Ms, _) in syn.SHAPES for M in Ms]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name,M", CASES)
def test_gemv_workload_shapes(w4, name, M, path):
    _, K, N, _, srange = syn.shape(name)
    p = syn.make_problem(f"{name}.M{M}", K, N, M, seed=0, scale_range=srange)
    got32, got16, _ = run_gemv(w4, p, path=path)
    splits = path_splits(w4, path, K, N)
    rows = sample_rows(N, np.random.default_rng(1)) if M * N * K > 2 ** 28 else np.arange(N)
    ref, refabs = oracle_rows(p, rows)
    mag, extra = bound_terms(w4, path, p, rows, refabs)
    tu.check_gemv(got32[:, rows], got16[:, rows], ref, mag, K, splits, f"{name} M={M} {path}",
                  extra)


# ---- edge cases ---------------------------------------------------------------------

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,K,N", [(1, 128, 1), (3, 128, 17), (8, 256, 200), (2, 1152, 1000),
                                   (7, 384, 48), (4, 18944, 40), (5, 17408, 33),
                                   (1, 640, 16), (6, 2048, 513), (1, 4096, 20000)])
def test_gemv_ragged_and_small(w4, M, K, N, path):
    p = syn.make_problem(f"edge.{M}.{K}.{N}", K, N, M, seed=2)
    got32, got16, _ = run_gemv(w4, p, path=path)
    ref, refabs = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, with_abs=True)
    splits = path_splits(w4, path, K, N)
    mag, extra = bound_terms(w4, path, p, None, refabs)
    tu.check_gemv(got32, got16, ref, mag, K, splits, f"edge {M},{K},{N} {path}", extra)


@pytest.mark.parametrize("M,K,N", [(3, 1024, 64037), (8, 1024, 64037), (4, 768, 70001)])
def test_gemv_persistent_grid(w4, M, K, N):
    """Products of several waves without a K split run persistent from three
    tokens on (each block takes row blocks in turn): oracle parity on sampled
    rows including the ragged last row block, and every token's result equal
    bit for bit to the single-token product, which runs one block per row
    block."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, splits, fold = w4.gemv_config(K, N)
    assert splits == 1 and (N + 127) // 128 > 3 * sms
    assert fold == (K // 128 >= 8)
    p = syn.make_problem(f"persist.{M}.{K}.{N}", K, N, M, seed=4)
    got32, got16, packed = run_gemv(w4, p)
    rows = sample_rows(N, np.random.default_rng(5))
    ref, refabs = oracle_rows(p, rows)
    mag, extra = bound_terms(w4, "cluster", p, rows, refabs)
    tu.check_gemv(got32[:, rows], got16[:, rows], ref, mag, K, 1, f"persistent {M},{K},{N}",
                  extra)
    _, _, _, x = tu.to_device(p)
    for r in range(M):
        one = packed.gemv_f32(x[r:r + 1].contiguous()).cpu().numpy()
        assert np.array_equal(one[0], got32[r]), r


def _scale_bf16(bits, k):
    """bf16 bit patterns times 2^k (exponent field moved by k; zeros stay)."""
    b = bits.astype(np.int32)
    e = (b >> 7) & 0xFF
    assert ((e == 0) | ((e + k > 0) & (e + k < 255))).all()
    return np.where(e == 0, b, b + (k << 7)).astype(bits.dtype)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [3, 6])
def test_gemv_x_dynamic_range(w4, path, M):
    """x far outside the fp16 range, tiny, zero and mixed within one group,
    and ordinary tokens with values below 2^-17: the folded fp16 path scales
    each token by a power of two into fp16 range, so the result stays within
    the bound (which counts the fp16 rounding of values more than 2^28 below
    their token's largest).  M = 3 and 6 take the two x prologues of the
    folded path."""
    K, N = 8192, 384
    p = syn.make_problem("xrange", K, N, M, seed=12)
    x = p.x.copy()
    x[0, 0:128] = _scale_bf16(x[0, 0:128], 40)          # |x| up to ~2^42
    x[0, 128:256] = _scale_bf16(x[0, 128:256], -60)     # a group ~2^-60 beside it
    x[0, 256:384] = 0                                   # an all-zero group
    x[1, 384:448] = _scale_bf16(x[1, 384:448], 30)      # 2^30 next to 2^-30 in one group
    x[1, 448:512] = _scale_bf16(x[1, 448:512], -30)
    x[2, ::37] = 0x3400                                 # 2^-23 in an ordinary token
    x[2, 5::41] = 0
    if M > 3:
        x[3, :] = _scale_bf16(x[3, :], -100)            # a whole token tiny
        x[4, :] = _scale_bf16(x[4, :], -3)              # largest ~0.4
        x[5, :] = _scale_bf16(x[5, :], -6)              # largest ~0.05
    p = syn.Problem(p.name, M, K, N, p.qweight, p.scales, p.zeros, x)
    got32, got16, _ = run_gemv(w4, p, path=path)
    assert np.isfinite(got32).all()
    ref, refabs = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, with_abs=True)
    mag, extra = bound_terms(w4, path, p, None, refabs)
    tu.check_gemv(got32, got16, ref, mag, K, path_splits(w4, path, K, N), f"x range {path}",
                  extra)


def test_split_paths_covered(w4):
    cfg = [w4.gemv_config(K, N) for (_, K, N, _, _) in syn.SHAPES]
    splits = {c[1] for c in cfg}
    assert 1 in splits and any(s > 1 for s in splits), splits
    assert {c[2] for c in cfg} == {False, True}, cfg


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("K", [1024, 8192])
def test_q_equals_z_gives_zero(w4, path, K):
    """q = z everywhere: y = 0, exactly where the tensor-core operand is q - z,
    within the fp32 bound of (128 + z) sum x - (128 + z) sum x where the zero
    point is folded (the cluster split at K = 8192)."""
    M, N = 4, 100
    p = syn.make_problem("qz", K, N, M, seed=4)
    z = p.zeros
    q = np.repeat(z, 128, axis=1).astype(np.uint32)
    words = np.zeros((N, K // 8), np.uint32)
    for j in range(8):
        words |= q[:, j::8] << np.uint32(4 * j)
    p.qweight = words
    got32, got16, _ = run_gemv(w4, p, path=path)
    if not folds(w4, path, K, N):
        assert np.all(got32 == 0.0) and np.all((got16 & 0x7FFF) == 0)
    else:
        n = 8 + K // 128 + path_splits(w4, path, K, N) + 1 + tu.FOLD_EXTRA_STEPS
        assert (np.abs(got32) <= n * 2.0 ** -23 * tu.folded_abs(p)).all()
        assert np.array_equal(got16, oracle.bf16_rne(got32))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("Kd", [256, 8192])
def test_one_hot_and_identity(w4, path, Kd):
    """One-hot x: exact on both splits and both arithmetics (a single nonzero
    product per output).  Identity pattern (q - z = 1 on the diagonal): exact
    where the operand is q - z, within the fp32 bound where the zero point is
    folded."""
    M, K, N = 8, 512, 96
    if Kd == 8192:
        K = 8192
        ks = [0, 1, 127, 128, 2000, 4095, 6000, 8191]
    else:
        ks = [0, 1, 127, 128, 255, 300, 448, 511]
    p = syn.make_problem("onehot", K, N, M, seed=5)
    x = np.zeros((M, K), np.uint16)
    vals = [0x3F80, 0xC040, 0x3E20, 0x4109, 0xBF00, 0x3F81, 0x4000, 0xC2F6]
    for m in range(M):
        x[m, ks[m]] = vals[m]
    p.x = x
    got32, _, _ = run_gemv(w4, p, path=path)
    ref = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N)
    assert np.array_equal(got32, ref.astype(np.float32))
    # identity pattern: q - z = 1 on the diagonal, 0 elsewhere; y = s * x exactly
    Nd = 256
    z = np.random.default_rng(6).integers(0, 15, size=(Nd, Kd // 128))
    q = np.repeat(z, 128, axis=1)
    for n in range(Nd):
        q[n, n] = z[n, n // 128] + 1
    words = np.zeros((Nd, Kd // 8), np.uint32)
    for j in range(8):
        words |= q[:, j::8].astype(np.uint32) << np.uint32(4 * j)
    pi = syn.make_problem("ident", Kd, Nd, 3, seed=7)
    pi.qweight, pi.zeros = words, z.astype(np.uint8)
    got32, _, _ = run_gemv(w4, pi, path=path)
    ref = oracle.gemv_f64(pi.qweight, pi.scales, pi.zeros, pi.x, 3, Kd, Nd)
    if not folds(w4, path, Kd, Nd):
        assert np.array_equal(got32, ref.astype(np.float32))
    else:
        n = 8 + Kd // 128 + path_splits(w4, path, Kd, Nd) + 1 + tu.FOLD_EXTRA_STEPS
        assert (np.abs(got32 - ref) <= n * 2.0 ** -23 * tu.folded_abs(pi)).all()


@pytest.mark.parametrize("path", PATHS)
def test_linearity_power_of_two_exact(w4, path):
    M, K, N = 3, 3584, 300
    p = syn.make_problem("lin", K, N, M, seed=8)
    a32, _, packed = run_gemv(w4, p, path=path)
    xf = (p.x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0)
    p2 = syn.Problem("lin2", M, K, N, p.qweight, p.scales, p.zeros,
                     (xf.view(np.uint32) >> 16).astype(np.uint16))
    b32, _, _ = run_gemv(w4, p2, packed, path=path)
    assert np.array_equal(b32, 2 * a32)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("K,N", [(18944, 3584), (3584, 37888)])
def test_determinism_and_batch_invariance(w4, path, K, N):
    p = syn.make_problem("det", K, N, 8, seed=9)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack(qw, sc, zp, K, N)
    ws = w4.workspace(K, N) if path == "ws" else None
    first = packed.gemv_f32(x, workspace=ws).cpu()
    for _ in range(50):
        assert torch.equal(packed.gemv_f32(x, workspace=ws).cpu(), first)
    for r in (0, 3, 7):
        one = packed.gemv_f32(x[r:r + 1].contiguous(), workspace=ws).cpu()
        assert torch.equal(one[0], first[r])
    five = packed.gemv_f32(x[:5].contiguous(), workspace=ws).cpu()
    assert torch.equal(five, first[:5])


@pytest.mark.parametrize("path", PATHS)
def test_graph_capture_replay(w4, path):
    K, N, M = 3584, 4608, 1
    p = syn.make_problem("graph", K, N, M, seed=10)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack(qw, sc, zp, K, N)
    ws = w4.workspace(K, N) if path == "ws" else None
    y_eager = packed.gemv(x, workspace=ws)
    y = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        packed.gemv(x, y, workspace=ws)            # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        packed.gemv(x, y, workspace=ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)


# The capture below records nothing on purpose (the repack refuses to run
# under capture), so torch's "graph is empty" warning is expected.
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_repack_rejects_bad_zero_and_capture(w4):
    K, N = 256, 32
    p = syn.make_problem("badz", K, N, 1, seed=11)
    p.zeros[5, 1] = 16
    qw, sc, zp, _ = tu.to_device(p)
    with pytest.raises(w4.W4Error) as e:
        w4.pack(qw, sc, zp, K, N)
    assert e.value.status == w4.Status.INVALID_ARG
    # a stream being captured: repack synchronises, so it refuses
    p.zeros[5, 1] = 3
    qw, sc, zp, _ = tu.to_device(p)
    qb, sb, zb = w4.repacked_sizes(K, N)
    bufs = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in (qb, sb, zb)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            with pytest.raises(w4.W4Error) as e2:
                w4.repack(qw, sc, zp, K, N, *bufs, stream=s)
    assert e2.value.status == w4.Status.UNSUPPORTED


def test_header_checked(w4):
    K, N = 384, 64
    p = syn.make_problem("hdr", K, N, 1, seed=12)
    qw, sc, zp, _ = tu.to_device(p)
    packed = w4.pack(qw, sc, zp, K, N)
    hdr = packed.qweight[:128].cpu().numpy().tobytes()
    w4.check_header(hdr, K, N)
    with pytest.raises(w4.W4Error):
        w4.check_header(hdr, K, N + 16)


def test_argument_errors_on_device(w4):
    K, N = 256, 32
    p = syn.make_problem("args", K, N, 2, seed=13)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack(qw, sc, zp, K, N)
    y = torch.empty((2, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.gemv(packed.qweight, packed.scales, packed.zeros, x, y, 9, K, N)
    assert e.value.status == w4.Status.UNSUPPORTED
    with pytest.raises(w4.W4Error) as e:
        w4.gemv(packed.qweight, packed.scales, packed.zeros, x, y, 2, 200, N)
    assert e.value.status == w4.Status.INVALID_ARG
    short = torch.zeros(w4.gemv_workspace_bytes(K, N) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.gemv_ws(packed.qweight, packed.scales, packed.zeros, x, y, 2, K, N, short)
    assert e.value.status == w4.Status.INVALID_ARG


def test_ws_and_cluster_paths_agree(w4):
    """Both splits compute the same sums in a different order: they differ by
    no more than the sum of the two paths' fp32 rounding bounds."""
    K, N, M = 3584, 37888, 2
    p = syn.make_problem("paths", K, N, M, seed=14)
    a32, _, packed = run_gemv(w4, p, path="cluster")
    b32, _, _ = run_gemv(w4, p, packed, path="ws")
    rows = sample_rows(N, np.random.default_rng(15))
    _, refabs = oracle_rows(p, rows)
    n_cl = 8 + K // 128 + path_splits(w4, "cluster", K, N) + 1 + tu.FOLD_EXTRA_STEPS
    n_ws = 8 + K // 128 + K // 128 + 1
    bound = 2.0 ** -23 * (n_cl * tu.folded_abs(p, rows) + n_ws * refabs)
    assert (np.abs(a32[:, rows].astype(np.float64) - b32[:, rows]) <= bound).all()


# ---- nothing is written outside y ---------------------------------------------------

@pytest.mark.parametrize("path,M,K,N", [("cluster", 1, 3584, 3584), ("cluster", 8, 18944, 200),
                                        ("cluster", 1, 3584, 37888), ("cluster", 4, 1024, 64037),
                                        ("ws", 3, 3584, 1000), ("swiglu", 2, 1024, 333)])
def test_no_write_outside_y(w4, path, M, K, N):
    """The output is written exactly: y sits between two 4 KB guard bands of a
    sentinel pattern, which must be unchanged after bf16 and fp32 calls (the
    cluster split at one-wave, tall-K and persistent launch shapes, the
    workspace split, the SwiGLU product with a ragged last tile)."""
    rows = 2 * N if path == "swiglu" else N
    p = syn.make_problem(f"guard.{path}.{M}.{K}.{N}", K, rows, M, seed=16)
    qw, sc, zp, x = tu.to_device(p)
    packed = w4.pack_swiglu(qw, sc, zp, K, N) if path == "swiglu" else w4.pack(qw, sc, zp, K, N)
    ws = w4.workspace(K, N) if path == "ws" else None
    guard = 4096
    for esize, fn in ((2, "gemv"), (4, "gemv_f32")):
        nbytes = M * N * esize
        buf = torch.full((2 * guard + nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
        y = buf[guard:guard + nbytes].view(torch.bfloat16 if esize == 2 else torch.float32)
        y = y.view(M, N)
        if path == "swiglu":
            getattr(packed, fn)(x, y)
        else:
            getattr(packed, fn)(x, y, workspace=ws)
        torch.cuda.synchronize()
        host = buf.cpu().numpy()
        assert (host[:guard] == 0x5A).all(), f"{path} {fn}: write before y"
        assert (host[guard + nbytes:] == 0x5A).all(), f"{path} {fn}: write after y"
        assert not (host[guard:guard + nbytes] == 0x5A).all(), f"{path} {fn}: y not written"
