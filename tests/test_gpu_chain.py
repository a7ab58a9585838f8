"""Dependent chains of W4 products, as single-request decode runs them: one
CUDA graph per step in which every product's input x is the output y of the
product before it, launched with programmatic dependent launch so that each
kernel starts (and requests its first weight records) while the previous one
is still finishing ("qengine", section "How it works": one CUDA graph per
decode step, each kernel starting its loads while the previous one drains).

What must hold under that overlap:
  * read after write -- a product reads x only once the product that writes
    it has completed (the kernels wait on griddepcontrol before touching x);
  * write after read -- a product writes y only once the product that reads
    that buffer as its x has completed (the kernels wait again before their
    first store).
Weights never depend on an earlier kernel, which is why they may be requested
before the wait; the graphs below check that this early issue changes nothing.

Each chain is captured once and replayed several times.  Before every replay
all activation buffers except the chain's input are filled with bfloat16 NaN,
so a read that overtakes its producer sees NaN (or, if it sees stale values
from an earlier replay, the ping-pong comparison below differs).  Every
step's output is compared with the oracle applied to the GPU's own bfloat16
output of the previous step, so errors do not compound ("CodeAlign-Runtime",
section "Benchmarking Methodology": correctness accompanies every speed run):
the chained output must equal, bit for bit, the same product run alone on
that input, whose fp32 result must match the oracle within the library's
tolerances.

Chains (launch shapes asserted through w4_gemv_plan):
  * square: o-shaped 3584 -> 3584 products (K split over a cluster, exact
    operand, one wave capped at two blocks per SM, overlapped), M = 1 and 8;
  * mlp: the 7B gated MLP, gate/up + SwiGLU 3584 -> 18944 then down
    18944 -> 3584, twice (zero point folded), M = 1 and 8;
  * persistent: three 1024 -> 65536 products at M = 3 and 8, each reading
    the first M x 1024 values of the previous output as its x (several-wave
    products on the persistent grid, which store row block by row block).
Each runs once with a distinct buffer per step (read after write; every step
checked) and once with two buffers used in turn (step i + 1 writes the buffer
step i reads: write after read); the two runs' last outputs must be
bit-identical.
"""
import numpy as np
import pytest

import oracle
from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu
from tests.test_gpu_swiglu import bound as swiglu_bound
from tests.test_gpu_swiglu import check as swiglu_check

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BF16_NAN = 0x7FC0


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


class Step:
    """One product of a chain: an N x K weight (plain) or a fused [2I, K]
    gate/up weight (swiglu, output width I)."""

    def __init__(self, w4, name, K, out, swiglu=False):
        self.name, self.K, self.out, self.swiglu = name, K, out, swiglu
        rows = 2 * out if swiglu else out
        self.qw, self.sc, self.zp = syn.make_weights(name, K, rows, seed=21)
        dq = torch.from_numpy(self.qw.view(np.int32)).cuda()
        ds = torch.from_numpy(self.sc.view(np.int16)).cuda()
        dz = torch.from_numpy(self.zp).cuda()
        self.packed = (w4.pack_swiglu(dq, ds, dz, K, out) if swiglu
                       else w4.pack(dq, ds, dz, K, out))

    def launch(self, x, y, stream):
        self.packed.gemv(x, y, stream=stream)

    def check(self, w4, xbits, got16, M, rng, what):
        """The chained bf16 output of this step must be bit-identical to the
        same product run alone on the same x (the GPU's bf16 output of the
        step before), rounded to bf16; and that product's fp32 output must
        match the oracle on the same x within the library's tolerances."""
        x = tu.x_to_device(xbits)
        got32 = self.packed.gemv_f32(x).cpu().numpy()
        assert np.isfinite(got32).all(), f"{what}: non-finite output"
        assert np.array_equal(got16, oracle.bf16_rne(got32)), \
            f"{what}: the chained output differs from the same product run alone"
        N = 2 * self.out if self.swiglu else self.out
        p = syn.Problem(self.name, M, self.K, N, self.qw, self.sc, self.zp, xbits)
        cols = (np.arange(self.out) if self.out <= 2048 else np.unique(np.concatenate(
            [np.arange(64), np.arange(self.out - 64, self.out),
             rng.choice(self.out, 1024, replace=False)])))
        if self.swiglu:
            y, b = swiglu_bound(w4, p, self.out, cols)
            swiglu_check(got32[:, cols], got16[:, cols], y, b, what)
            return
        ref, refabs = oracle.gemv_rows_f64(p.qweight, p.scales, p.zeros, p.x, M, p.K, p.N,
                                           cols, with_abs=True)
        _, S, fold = w4.gemv_config(p.K, p.N)
        mag = tu.folded_abs(p, cols) if fold else refabs
        tu.check_gemv(got32[:, cols], got16[:, cols], ref, mag, p.K, S, what,
                      tu.FOLD_EXTRA_STEPS if fold else 0)


def build_chain(w4, kind):
    if kind == "square":
        return [Step(w4, f"chain.sq{i}", 3584, 3584) for i in range(6)]
    if kind == "mlp":
        out = []
        for i in range(2):
            out.append(Step(w4, f"chain.gu{i}", 3584, 18944, swiglu=True))
            out.append(Step(w4, f"chain.dn{i}", 18944, 3584))
        return out
    if kind == "persistent":
        return [Step(w4, f"chain.p{i}", 1024, 65536) for i in range(3)]
    raise ValueError(kind)


def run_chain(steps, M, x0bits, pingpong, replays=3):
    """Capture the chain in one graph, replay it `replays` times (activation
    buffers NaN-filled before each), return the bf16 outputs of every step
    (distinct buffers) or of the last two steps (ping-pong)."""
    x0 = tu.x_to_device(x0bits)
    if pingpong:
        width = max(s.out for s in steps)
        bufs = [torch.empty(M * width, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        # step 0 reads x0 and writes bufs[0]; step i reads bufs[(i-1)%2], writes bufs[i%2]
        outs = [bufs[i % 2][:M * steps[i].out].view(M, steps[i].out) for i in range(len(steps))]
    else:
        bufs = [torch.empty((M, s.out), dtype=torch.bfloat16, device="cuda") for s in steps]
        outs = bufs
    # step i reads the first M x K values of step i - 1's output as its x
    ins = [x0] + [o.reshape(-1)[:M * s.K].view(M, s.K) for o, s in zip(outs[:-1], steps[1:])]
    stream = torch.cuda.Stream()

    def calls():
        for s, xi, yi in zip(steps, ins, outs):
            s.launch(xi, yi, stream)

    with torch.cuda.stream(stream):
        calls()                       # warm-up outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    results = []
    for _ in range(replays):
        for b in bufs:
            b.view(torch.int16).fill_(BF16_NAN)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        if pingpong:
            results.append([tu.bf16_bits(outs[-2]), tu.bf16_bits(outs[-1])])
        else:
            results.append([tu.bf16_bits(o) for o in outs])
    return results


CHAIN_CASES = [("square", 1), ("square", 8), ("mlp", 1), ("mlp", 8), ("persistent", 3),
               ("persistent", 8)]


def assert_launch_shapes(w4, kind, steps, M):
    plans = [w4.gemv_plan(M, s.K, 16 * ((s.out + 7) // 8) if s.swiglu else s.out)
             for s in steps]
    # every step after the first may start early (programmatic dependent launch)
    assert all(p["overlap"] for p in plans[1:]), plans
    if kind == "square":
        assert all(p["k_splits"] > 1 and not p["persistent"] for p in plans), plans
    if kind == "mlp":
        assert all(p["zero_point_folded"] for p in plans), plans
    if kind == "persistent":
        assert all(p["persistent"] for p in plans), plans


@pytest.mark.parametrize("kind,M", CHAIN_CASES)
def test_dependent_chain(w4, kind, M):
    steps = build_chain(w4, kind)
    assert_launch_shapes(w4, kind, steps, M)
    x0bits = syn.make_x(f"chain.{kind}.x0", M, steps[0].K, seed=21)
    distinct = run_chain(steps, M, x0bits, pingpong=False)
    # every replay bit-identical (determinism across replays)
    for r in distinct[1:]:
        for a, b in zip(distinct[0], r):
            assert np.array_equal(a, b)
    rng = np.random.default_rng(22)
    outs = distinct[0]
    xin = x0bits
    for i, (s, y) in enumerate(zip(steps, outs)):
        s.check(w4, xin, y, M, rng, f"{kind} M={M} step {i} ({s.name})")
        if i + 1 < len(steps):
            xin = y.reshape(-1)[:M * steps[i + 1].K].reshape(M, steps[i + 1].K)
    # write after read: the ping-pong chain ends in the same bits
    pp = run_chain(steps, M, x0bits, pingpong=True)
    for r in pp:
        assert np.array_equal(r[0], outs[-2]), f"{kind} M={M}: ping-pong step {len(steps) - 2}"
        assert np.array_equal(r[1], outs[-1]), f"{kind} M={M}: ping-pong last step"
