"""The seeded input generator: reproducible, independent streams, right ranges."""
import numpy as np

from int4_weight_only_w4_gb300 import synthetic as syn


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 started from state 0 (Vigna's splitmix64.c)
    z = np.arange(1, 5, dtype=np.uint64) * np.uint64(syn.GAMMA)
    got = [int(v) for v in syn._mix(z)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                   0x06C45D188009454F, 0xF88BB8A8724C81EC]


def test_counter_slices_and_threads_agree():
    full = syn.u64(0, "t", (1 << 23) + 5)           # threaded path
    part = syn.u64(0, "t", 1000, start=(1 << 22) - 3)
    assert np.array_equal(full[(1 << 22) - 3:(1 << 22) + 997], part)
    assert not np.array_equal(syn.u64(0, "t", 64), syn.u64(0, "u", 64))
    assert not np.array_equal(syn.u64(0, "t", 64), syn.u64(1, "t", 64))


def test_problem_ranges_and_reproducibility():
    p = syn.make_problem("x", 512, 64, 3, seed=0, scale_range=(0.0005, 0.01))
    q = syn.make_problem("x", 512, 64, 3, seed=0, scale_range=(0.0005, 0.01))
    for a in ("qweight", "scales", "zeros", "x"):
        assert np.array_equal(getattr(p, a), getattr(q, a))
    assert p.qweight.shape == (64, 64) and p.qweight.dtype == np.uint32
    assert p.scales.shape == (64, 4) and p.zeros.shape == (64, 4) and p.x.shape == (3, 512)
    s = p.scales.view(np.float16).astype(np.float64)
    assert s.min() >= 0.0005 * (1 - 2 ** -10) and s.max() <= 0.01 * (1 + 2 ** -10)
    assert p.zeros.max() <= 15


def test_distributions():
    q = syn.uniform_words(0, "w", (4096,))
    nib = np.concatenate([(q >> np.uint32(4 * j)) & np.uint32(15) for j in range(8)])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    x = syn.normal_bf16(0, "n", (200000,))
    xf = (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert abs(xf.mean()) < 0.01 and abs(xf.std() - 1) < 0.01
