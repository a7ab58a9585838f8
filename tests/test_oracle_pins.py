"""Pins for the CPU oracle: checks against things other than the oracle itself.

Every expected value here comes from (a) a worked example in tests/golden/
derived by hand from the format's definition, (b) exact rational arithmetic
(fractions.Fraction) on tiny inputs built from *unpacked* integers, so a
nibble-order, index, sign or transposition mistake in the oracle shows up,
(c) closed forms (one-hot x, identity-pattern W, q == z), or (d) a library's
own rounding (numpy binary16, torch bfloat16).
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- helpers written for the tests (independent of the oracle) -------------

def pack_rows(q):
    """q[N][K] ints 0..15 -> uint32 [N][K/8], nibble j of word w = k 8w+j."""
    q = np.asarray(q, dtype=np.uint32)
    N, K = q.shape
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        words |= q[:, j::8] << np.uint32(4 * j)
    return words


def half_value(bits):
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


def bf16_value(bits):
    return Fraction(float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0]))


def exact_y(q, z, s_bits, x_bits):
    """Exact y[M][N] from unpacked q[N][K], z[N][G], scale bits, x bits."""
    N, K = len(q), len(q[0])
    M = len(x_bits)
    s = [[half_value(b) for b in row] for row in s_bits]
    xv = [[bf16_value(b) for b in row] for row in x_bits]
    y = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // 128
                acc += (int(q[n][k]) - int(z[n][g])) * s[n][g] * xv[m][k]
            y[m][n] = acc
    return y


def random_case(rng, M, K, N, scale_lo=0.001, scale_hi=0.02):
    G = K // 128
    q = rng.integers(0, 16, size=(N, K), dtype=np.int64)
    z = rng.integers(0, 16, size=(N, G), dtype=np.int64)
    s_bits = rng.uniform(scale_lo, scale_hi, size=(N, G)).astype(np.float16).view(np.uint16)
    x_f = rng.standard_normal(size=(M, K)).astype(np.float32)
    x_bits = (x_f.view(np.uint32) >> 16).astype(np.uint16)     # truncation: any bf16 will do
    return q, z, s_bits, x_bits


def read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append(vals)
    return out


# ---- worked examples --------------------------------------------------------

def test_golden_nibble_order():
    fx = read_fixture("nibble_order.txt")
    K, N, M = (int(fx[k][0][0]) for k in ("K", "N", "M"))
    qweight = np.array([[int(w, 16) for w in fx["qweight"][0]]], dtype=np.uint32)
    scales = np.array([[int(fx["scales"][0][0], 16)]], dtype=np.uint16)
    zeros = np.array([[int(fx["zeros"][0][0])]], dtype=np.uint8)
    x = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        x[m, m] = int(fx["x_onehot_value"][0][0], 16)
    y = oracle.gemv_f64(qweight, scales, zeros, x, M, K, N)
    want = np.array([float(v) for v in fx["y"][0]])
    assert np.array_equal(y[:, 0], want)


def test_golden_group_index():
    fx = read_fixture("group_index.txt")
    K, N, M = (int(fx[k][0][0]) for k in ("K", "N", "M"))
    qweight = np.empty((N, K // 8), dtype=np.uint32)
    qweight[0] = int(fx["row0_word"][0][0], 16)
    qweight[1] = int(fx["row1_word"][0][0], 16)
    scales = np.array([int(v, 16) for v in fx["scales"][0]], dtype=np.uint16).reshape(N, 2)
    zeros = np.array([int(v) for v in fx["zeros"][0]], dtype=np.uint8).reshape(N, 2)
    x = np.empty((M, K), dtype=np.uint16)
    x[:, :128] = int(fx["x_lo"][0][0], 16)
    x[:, 128:] = int(fx["x_hi"][0][0], 16)
    y = oracle.gemv_f64(qweight, scales, zeros, x, M, K, N)
    assert np.array_equal(y[0], [float(v) for v in fx["y"][0]])
    w16 = oracle.dequant_f16(qweight, scales, zeros, K, N)
    for r, key in enumerate(("w16_row0", "w16_row1")):
        lo, hi = (int(v, 16) for v in fx[key][0])
        assert np.all(w16[r, :128] == lo) and np.all(w16[r, 128:] == hi)


def test_golden_dequant_rounding():
    fx = read_fixture("dequant_rounding.txt")
    s = int(fx["scale"][0][0], 16)
    for q, z, want in fx["case"]:
        q, z, want = int(q), int(z), int(want, 16)
        qweight = np.full((1, 16), 0, dtype=np.uint32)
        qweight[0, 0] = q                     # nibble 0 of word 0 is k = 0
        scales = np.array([[s]], dtype=np.uint16)
        zeros = np.array([[z]], dtype=np.uint8)
        w16 = oracle.dequant_f16(qweight, scales, zeros, 128, 1)
        assert int(w16[0, 0]) == want, (q, z, hex(int(w16[0, 0])), hex(want))


def test_golden_symmetric_special_case():
    fx = read_fixture("symmetric_nibbles.txt")
    pages_word = int(fx["pages_word"][0][0], 16)
    canon_word = int(fx["canonical_word"][0][0], 16)
    signed = [int(v) for v in fx["signed"][0]]
    # the pages' reading: mask the nibble, sign-extend when bit 3 is set
    for k in range(8):
        nib = (pages_word >> (4 * k)) & 0xF
        v = nib - 16 if nib & 0x8 else nib
        assert v == signed[k]
        assert ((canon_word >> (4 * k)) & 0xF) == nib ^ 0x8
    qweight = np.full((1, 16), 0x88888888, dtype=np.uint32)
    qweight[0, 0] = canon_word
    scales = np.array([[0x3C00]], dtype=np.uint16)
    zeros = np.array([[8]], dtype=np.uint8)
    x = np.zeros((1, 128), dtype=np.uint16)
    x[0, :8] = 0x3F80
    y = oracle.gemv_f64(qweight, scales, zeros, x, 1, 128, 1)
    assert y[0, 0] == float(fx["y"][0][0])


# ---- exact rational brute force ---------------------------------------------

@pytest.mark.parametrize("M,K,N,seed", [(8, 128, 8, 0), (2, 256, 3, 1), (3, 384, 5, 2),
                                        (1, 128, 1, 3), (5, 256, 4, 4)])
def test_bruteforce_exact(M, K, N, seed):
    rng = np.random.default_rng(seed)
    q, z, s_bits, x_bits = random_case(rng, M, K, N)
    qweight = pack_rows(q)
    y, yabs = oracle.gemv_f64(qweight, s_bits, z.astype(np.uint8), x_bits, M, K, N,
                              with_abs=True)
    ex = exact_y(q.tolist(), z.tolist(), s_bits.tolist(), x_bits.tolist())
    for m in range(M):
        for n in range(N):
            # recursive fp64 summation of exact products: |err| <= (K-1) u sum|p|
            bound = (K - 1) * 2.0 ** -53 * yabs[m, n]
            assert abs(Fraction(y[m, n]) - ex[m][n]) <= Fraction(bound), (m, n)


def test_rows_subset_matches_bruteforce():
    rng = np.random.default_rng(11)
    M, K, N = 2, 256, 9
    q, z, s_bits, x_bits = random_case(rng, M, K, N)
    qweight = pack_rows(q)
    rows = [8, 0, 5, 5]
    y = oracle.gemv_rows_f64(qweight, s_bits, z.astype(np.uint8), x_bits, M, K, N, rows)
    ex = exact_y(q.tolist(), z.tolist(), s_bits.tolist(), x_bits.tolist())
    for m in range(M):
        for i, r in enumerate(rows):
            assert abs(Fraction(y[m, i]) - ex[m][r]) <= Fraction(1e-12)


def test_dequant_f32_exact_and_f16_rounding():
    # exhaustive q, z with scales over the binary16 range (normal, subnormal,
    # large enough that the product overflows binary16)
    scale_bits = [0x3C00, 0x2E66, 0x1400, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0x5A00, 0x3555]
    K, N = 128, len(scale_bits) * 16
    q = np.zeros((N, K), dtype=np.int64)
    z = np.zeros((N, 1), dtype=np.int64)
    s = np.zeros((N, 1), dtype=np.uint16)
    row = 0
    for sb in scale_bits:
        for zz in range(16):
            q[row, :16] = np.arange(16)
            q[row, 16:] = zz
            z[row, 0] = zz
            s[row, 0] = sb
            row += 1
    qweight = pack_rows(q)
    w32 = oracle.dequant_f32(qweight, s, z.astype(np.uint8), K, N)
    w16 = oracle.dequant_f16(qweight, s, z.astype(np.uint8), K, N)
    for r in range(N):
        sv = half_value(int(s[r, 0]))
        for k in range(K):
            exact = (int(q[r, k]) - int(z[r, 0])) * sv
            assert Fraction(float(w32[r, k])) == exact
            with np.errstate(over="ignore"):
                want = np.float64(float(exact)).astype(np.float16).view(np.uint16)
            assert int(w16[r, k]) == int(want), (r, k)


# ---- closed forms -------------------------------------------------------------

def test_q_equals_z_gives_zero():
    rng = np.random.default_rng(5)
    M, K, N = 3, 512, 7
    z = rng.integers(0, 16, size=(N, K // 128))
    q = np.repeat(z, 128, axis=1)
    s = rng.uniform(0.001, 0.02, size=(N, K // 128)).astype(np.float16).view(np.uint16)
    x = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y = oracle.gemv_f64(pack_rows(q), s, z.astype(np.uint8), x, M, K, N)
    assert np.all(y == 0.0)


def test_linearity():
    rng = np.random.default_rng(6)
    M, K, N = 2, 384, 6
    q, z, s, _ = random_case(rng, M, K, N)
    qw = pack_rows(q)
    # integer-valued x so that x1 + x2 and 2 * x1 are exact in bfloat16
    x1i = rng.integers(-100, 101, size=(M, K)).astype(np.float32)
    x2i = rng.integers(-100, 101, size=(M, K)).astype(np.float32)
    bf = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y1 = oracle.gemv_f64(qw, s, z.astype(np.uint8), bf(x1i), M, K, N, with_abs=True)
    y2 = oracle.gemv_f64(qw, s, z.astype(np.uint8), bf(x2i), M, K, N)
    y12 = oracle.gemv_f64(qw, s, z.astype(np.uint8), bf(x1i + x2i), M, K, N)
    y1x2 = oracle.gemv_f64(qw, s, z.astype(np.uint8), bf(2 * x1i), M, K, N)
    assert np.array_equal(y1x2, 2 * y1[0])
    assert np.allclose(y12, y1[0] + y2, rtol=0, atol=1e-9 * max(1.0, np.abs(y1[1]).max()))


def test_one_hot_x_exact():
    rng = np.random.default_rng(7)
    M, K, N = 4, 512, 10
    q, z, s, _ = random_case(rng, M, K, N)
    qw = pack_rows(q)
    ks = [0, 131, 300, 511]
    xval = [0x3F80, 0xC040, 0x3E20, 0x4109]     # 1, -3, 0.15625, 8.5625
    x = np.zeros((M, K), dtype=np.uint16)
    for m in range(M):
        x[m, ks[m]] = xval[m]
    y = oracle.gemv_f64(qw, s, z.astype(np.uint8), x, M, K, N)
    for m in range(M):
        g = ks[m] // 128
        for n in range(N):
            want = (int(q[n, ks[m]]) - int(z[n, g])) * half_value(int(s[n, g])) * bf16_value(xval[m])
            assert Fraction(y[m, n]) == want
            assert float(np.float32(y[m, n])) == float(want)   # exact in fp32 too


def test_identity_pattern_exact():
    K = N = 256
    M = 3
    rng = np.random.default_rng(8)
    z = rng.integers(0, 15, size=(N, K // 128))
    q = np.repeat(z, 128, axis=1)
    for n in range(N):
        q[n, n] = z[n, n // 128] + 1            # q - z = 1 on the diagonal only
    s = np.full((N, K // 128), 0x4000, dtype=np.uint16)   # 2.0
    x = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y = oracle.gemv_f64(pack_rows(q), s, z.astype(np.uint8), x, M, K, N)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(y, 2.0 * xv)


def test_symmetric_special_case_random():
    """z = 8 and nibble XOR 8 reproduce a direct signed-INT4 evaluation."""
    rng = np.random.default_rng(9)
    M, K, N = 2, 256, 5
    v = rng.integers(-8, 8, size=(N, K))
    s = rng.uniform(0.001, 0.02, size=(N, K // 128)).astype(np.float16).view(np.uint16)
    x = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    nib = v & 0xF                                # two's-complement nibbles (pages)
    q = nib ^ 0x8                                # offset binary
    zeros = np.full((N, K // 128), 8, dtype=np.uint8)
    y = oracle.gemv_f64(pack_rows(q), s, zeros, x, M, K, N)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sv = half_value(int(s[n, k // 128]))
                signed = int(nib[n, k]) - 16 if nib[n, k] & 0x8 else int(nib[n, k])
                acc += signed * sv * bf16_value(int(x[m, k]))
            assert abs(Fraction(y[m, n]) - acc) <= Fraction(1e-12)


# ---- number formats against library rounding ---------------------------------

def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_half_rne_matches_numpy():
    rng = np.random.default_rng(10)
    vals = list(rng.standard_normal(20000) * np.exp(rng.uniform(-25, 12, 20000)))
    # exact ties and boundaries
    vals += [1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65504.0, 65519.99, 65520.0, 2.0 ** -25,
             3 * 2.0 ** -26, 2.0 ** -24, 2.0 ** -14 - 2.0 ** -25, -0.0, 0.0, 1e9, -1e-9]
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.float64(v).astype(np.float16).view(np.uint16))
        assert oracle.double_to_half_rne(v) == want, v


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    bits = rng.integers(0, 2 ** 32, size=50000, dtype=np.uint64).astype(np.uint32)
    bits = bits[((bits >> 23) & 0xFF) != 0xFF]            # finite values
    ties = (rng.integers(0, 2 ** 16, size=2000).astype(np.uint32) << 16) | 0x8000
    bits = np.concatenate([bits, ties, np.array([0x7F7FFFFF, 0x7F7F8000], np.uint32)])
    bits = bits[((bits >> 23) & 0xFF) != 0xFF]            # NaN payloads are not pinned
    f = bits.view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne(f)
    assert np.array_equal(got, want)


def test_bf16_to_double_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_openmp_baseline_matches_oracle():
    """The OpenMP CPU baseline spreads the oracle's rows over threads without
    changing their arithmetic: bit-identical results, ragged shapes included."""
    from int4_weight_only_w4_gb300 import synthetic as syn
    assert oracle.omp_threads() >= 1
    for (M, K, N) in ((1, 128, 1), (3, 256, 17), (8, 1024, 200), (2, 4864, 33)):
        p = syn.make_problem(f"omp.{M}.{K}.{N}", K, N, M, seed=41)
        a = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N)
        b = oracle.gemv_f64_omp(p.qweight, p.scales, p.zeros, p.x, M, K, N)
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64)), (M, K, N)
