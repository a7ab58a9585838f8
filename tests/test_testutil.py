"""CPU checks of the test helpers' rounding-bound magnitudes."""
import numpy as np

import oracle
from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu


def test_folded_abs_matches_brute_force_and_dominates():
    M, K, N = 3, 384, 20
    p = syn.make_problem("fold", K, N, M, seed=21)
    got = tu.folded_abs(p)
    # brute force from the definition, one output at a time
    x = tu._bf16_to_f64(p.x)
    s = p.scales.view(np.float16).astype(np.float64)
    for m in range(M):
        for n in (0, 7, N - 1):
            tot = 0.0
            wsum = 0.0
            for g in range(K // 128):
                acc = 0.0
                z = int(p.zeros[n, g])
                for k in range(g * 128, g * 128 + 128):
                    q = (int(p.qweight[n, k // 8]) >> (4 * (k % 8))) & 0xF
                    first_half = (k % 16) < 8
                    acc += ((1024 if first_half else 64) + q) * abs(x[m, k])
                    acc += ((1024 if first_half else 64) + z) * abs(x[m, k])
                    wsum += abs(s[n, g]) * ((1024 if first_half else 64) + q)
                tot += abs(s[n, g]) * acc
            tot += wsum * max(np.abs(x[m]).max() * 2.0 ** -39, 2.0 ** -151) / 2.0 ** -23
            assert np.isclose(got[m, n], tot, rtol=1e-12)
    # (64 + q) >= |q - z|: the folded magnitudes bound the plain ones
    _, refabs = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N, with_abs=True)
    assert (got >= refabs).all()
