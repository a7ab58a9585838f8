"""Pins of the oracle's gate/up product with SwiGLU (w4o_gemv_swiglu_f64):
textbook values of the logistic function, the identity
silu(g) - silu(-g) = g, u = 0, and the pairing of gate row j with up row
I + j.  The matrix-vector products it composes are pinned in
test_oracle_pins.py."""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swiglu_points.txt")


def _weights(gs, us, K=128):
    """[2I, K] weights with s = 1, z = 8 and q - z = g (resp. u) at k = 0 and 0
    elsewhere, so that one-hot x at k = 0 gives gate = g, up = u exactly."""
    I = len(gs)
    q = np.full((2 * I, K), 8, np.int64)
    q[:I, 0] = 8 + np.array(gs)
    q[I:, 0] = 8 + np.array(us)
    words = np.zeros((2 * I, K // 8), np.uint32)
    for j in range(8):
        words |= q[:, j::8].astype(np.uint32) << np.uint32(4 * j)
    scales = np.full((2 * I, K // 128), 0x3C00, np.uint16)         # 1.0
    zeros = np.full((2 * I, K // 128), 8, np.uint8)
    x = np.zeros((1, K), np.uint16)
    x[0, 0] = 0x3F80                                                # 1.0
    return words, scales, zeros, x


def test_golden_points():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    gs = [int(r[0]) for r in rows]
    us = [int(r[1]) for r in rows]
    want = np.array([float(r[2]) for r in rows])
    qw, sc, zp, x = _weights(gs, us)
    y = oracle.gemv_swiglu_f64(qw, sc, zp, x, 1, 128, len(gs))[0]
    assert np.allclose(y, want, rtol=1e-14, atol=0), (y, want)


def test_odd_part_identity_and_zero_up():
    gs = [1, 2, 3, 5, 7]
    qw, sc, zp, x = _weights(gs + [-g for g in gs], [1] * 10)
    y = oracle.gemv_swiglu_f64(qw, sc, zp, x, 1, 128, 10)[0]
    assert np.allclose(y[:5] - y[5:], gs, rtol=1e-14)               # silu(g) - silu(-g) = g
    qw, sc, zp, x = _weights(gs, [0] * 5)
    assert np.all(oracle.gemv_swiglu_f64(qw, sc, zp, x, 1, 128, 5) == 0)


def test_gate_row_j_pairs_with_up_row_I_plus_j():
    """Distinct gates and ups: output j uses gate j and up j, not a neighbour."""
    gs = [1, -1, 2, 0]
    us = [1, 2, 3, 4]
    qw, sc, zp, x = _weights(gs, us)
    y = oracle.gemv_swiglu_f64(qw, sc, zp, x, 1, 128, 4)[0]
    sig = lambda t: 1.0 / (1.0 + np.exp(-t))                      # noqa: E731
    assert np.allclose(y, [0.7310585786300049, -0.5378828427399902, 3 * 1.761594155955765, 0],
                       rtol=1e-14)
    assert np.allclose(y, np.array(gs) * sig(np.array(gs, float)) * np.array(us), rtol=1e-14)
