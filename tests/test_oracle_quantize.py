"""Pins of the oracle's quantiser (w4o_quantize): a hand-worked fixture,
exact round trips of exactly representable groups, and error bounds.  The
dequantisation these tests use is itself pinned in test_oracle_pins.py."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_groups.txt")


def _groups():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, vals, exp, qs = [p.strip() for p in line.split("|")]
        gid, mode, period = head.split()
        scale, zero = exp.split()
        out.append((gid, int(mode), int(period), [float(v) for v in vals.split()],
                    int(scale, 16), int(zero), [int(v) for v in qs.split()]))
    return out


def _nibbles(qweight, K):
    q = np.empty((qweight.shape[0], K), np.int64)
    for j in range(8):
        q[:, j::8] = (qweight >> np.uint32(4 * j)) & 0xF
    return q


@pytest.mark.parametrize("case", _groups(), ids=lambda c: c[0])
def test_golden_groups(case):
    gid, mode, period, vals, scale, zero, qs = case
    K = 256                     # the group twice in one row: both groups must agree
    w = np.array([vals[k % period] for k in range(K)], np.float16).reshape(1, K)
    assert np.array_equal(w.astype(np.float64).ravel() % 1e9,
                          np.array([vals[k % period] for k in range(K)]) % 1e9)
    qw, sc, zp = oracle.quantize(w.view(np.uint16), K, 1, mode)
    assert list(sc[0]) == [scale, scale]
    assert list(zp[0]) == [zero, zero]
    assert list(_nibbles(qw, K)[0]) == [qs[k % period] for k in range(K)]


def test_exactly_representable_groups_round_trip():
    """w = (q - z) * s with q = 0 and q = 15 present and (q - z) * s exact in
    fp16: quantising returns the same q, z and s."""
    rng = np.random.default_rng(1)
    N, K = 64, 512
    G = K // 128
    s = np.ldexp(1.0 + rng.integers(0, 8, size=(N, G)) / 8.0, rng.integers(-12, 2, size=(N, G)))
    z = rng.integers(0, 16, size=(N, G))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::128] = 0
    q[:, 1::128] = 15
    w = (q - np.repeat(z, 128, axis=1)) * np.repeat(s, 128, axis=1)
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)
    qw, sc, zp = oracle.quantize(w16.view(np.uint16), K, N, oracle.QUANT_ASYM)
    assert np.array_equal(sc.view(np.float16).astype(np.float64), s)
    assert np.array_equal(zp, z)
    assert np.array_equal(_nibbles(qw, K), q)


@pytest.mark.parametrize("mode", [oracle.QUANT_ASYM, oracle.QUANT_SYM])
def test_error_bounds_and_ranges(mode):
    rng = np.random.default_rng(2 + mode)
    N, K = 96, 1024
    w = (rng.standard_normal((N, K)) * np.exp(rng.uniform(-6, 2, size=(N, 1)))).astype(np.float16)
    w[3, :128] = 0                              # an all-zero group
    w[4, 128:256] = 0.125                       # a constant group
    qw, sc, zp = oracle.quantize(w.view(np.uint16), K, N, mode)
    q = _nibbles(qw, K)
    assert q.min() >= 0 and q.max() <= 15
    if mode == oracle.QUANT_SYM:
        assert np.all(zp == 8)
    deq = oracle.dequant_f32(qw, sc, zp, K, N).astype(np.float64)
    s = np.repeat(sc.view(np.float16).astype(np.float64), 128, axis=1)
    err = np.abs(deq - w.astype(np.float64))
    # every weight within one step of the grid (clamping at the top of the
    # asymmetric range can cost up to one step; fp16 scale rounding a little)
    assert np.all(err <= s * (1.0 if mode == oracle.QUANT_ASYM else 0.5) * (1 + 2 ** -8) + 1e-30)
    assert np.all(deq[3, :128] == 0) and sc[3, 0] == 0
    # a constant positive group maps to the top code (its scale is rounded to
    # fp16, so the dequantised value is close to, not equal to, 0.125)
    assert np.all(q[4, 128:256] == 15)
    assert zp[4, 1] == (0 if mode == oracle.QUANT_ASYM else 8)


def test_modes_agree_on_the_symmetric_special_case():
    """Dequantised symmetric codes equal the pages' signed form
    clamp(rint(w / s), -8, 7) * s restated with numpy at the stored scale."""
    rng = np.random.default_rng(5)
    N, K = 8, 256
    w = rng.standard_normal((N, K)).astype(np.float16)
    qw, sc, zp = oracle.quantize(w.view(np.uint16), K, N, oracle.QUANT_SYM)
    s = np.repeat(sc.view(np.float16).astype(np.float32), 128, axis=1)
    code = np.clip(np.rint(w.astype(np.float32) / s), -8, 7)
    assert np.array_equal(_nibbles(qw, K) - 8, code.astype(np.int64))
