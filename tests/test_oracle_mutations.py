"""Plant plausible mistakes in a copy of the oracle and check that the pins catch
each one.  The copy is compiled into a temporary library; the real oracle source
is never changed."""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_quantize as qpins
from tests import test_oracle_swiglu as spins

MUTATIONS = {
    "sign of q - z": ("return (float)(q - z) * s;", "return (float)(z - q) * s;"),
    "zero point dropped": ("int z = zeros[gi];", "int z = 0;"),
    "nibble order reversed": ("(word >> (4 * (k % 8)))", "(word >> (4 * (7 - k % 8)))"),
    "x index reversed": ("x[(size_t)m * K + k]", "x[(size_t)m * K + (K - 1 - k)]"),
    "half exponent bias": ("e - 25", "e - 24"),
    "group index uses row stride K": ("(size_t)n * (size_t)G + (size_t)(k / W4O_GROUP)",
                                      "(size_t)(k / W4O_GROUP) * (size_t)G + (size_t)n % G"),
}

QUANT_MUTATIONS = {
    "asymmetric scale over 16 steps": ("(hi - lo) / 15.0f", "(hi - lo) / 16.0f"),
    "symmetric scale absmax / 8": ("amax / 7.0f", "amax / 8.0f"),
    "truncation instead of rounding": ("const float t = rintf(", "const float t = truncf("),
    "zero point sign flipped": ("rintf(-lo / s)", "rintf(lo / s)"),
    "zero left out of the range": ("float lo = 0.0f, hi = 0.0f, amax = 0.0f;",
                                   "float lo = 1e30f, hi = -1e30f, amax = 0.0f;"),
    "codes against the unrounded scale": ("const float t = rintf((float)w4o_half_to_double(wg[k]) / s);",
                                          "const float t = rintf((float)w4o_half_to_double(wg[k]) / s32);"),
}

QUANT_CHECKS = [
    lambda: [qpins.test_golden_groups(c) for c in qpins._groups()],
    qpins.test_exactly_representable_groups_round_trip,
    lambda: qpins.test_modes_agree_on_the_symmetric_special_case(),
]

SWIGLU_MUTATIONS = {
    "exp of +g": ("g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
    "up row off by one": ("K, I + j, m, &u, 0)", "K, I + j - (j > 0), m, &u, 0)"),
    "activation on the up product": ("g / (1.0 + exp(-g)) * u", "u / (1.0 + exp(-u)) * g"),
}

SWIGLU_CHECKS = [spins.test_golden_points, spins.test_odd_part_identity_and_zero_up,
                 spins.test_gate_row_j_pairs_with_up_row_I_plus_j]

PIN_CHECKS = [
    pins.test_golden_nibble_order,
    pins.test_golden_group_index,
    pins.test_golden_dequant_rounding,
    lambda: pins.test_bruteforce_exact(2, 256, 3, 1),
    pins.test_one_hot_x_exact,
]


def _caught(old, new, checks, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "w4_oracle.c")).read()
    assert old in src, "mutation site moved"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(path), "-lm"], check=True)
    saved_lib, saved_path, saved_build = oracle._lib, oracle._LIB_PATH, oracle.build
    try:
        oracle._lib = None
        oracle._LIB_PATH = str(so)
        oracle.build = lambda force=False, _p=str(so): _p  # noqa: E731 -- load the mutant
        caught = 0
        for check in checks:
            try:
                check()
            except AssertionError:
                caught += 1
        return caught
    finally:
        oracle._lib, oracle._LIB_PATH, oracle.build = saved_lib, saved_path, saved_build
        import importlib
        importlib.reload(oracle)


@pytest.mark.parametrize("name", sorted(SWIGLU_MUTATIONS))
def test_planted_swiglu_mistake_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = SWIGLU_MUTATIONS[name]
    assert _caught(old, new, SWIGLU_CHECKS, tmp_path) > 0, f"no pin caught mutation: {name}"


@pytest.mark.parametrize("name", sorted(QUANT_MUTATIONS))
def test_planted_quantiser_mistake_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = QUANT_MUTATIONS[name]
    assert _caught(old, new, QUANT_CHECKS, tmp_path) > 0, f"no pin caught mutation: {name}"


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "w4_oracle.c")).read()
    assert old in src, "mutation site moved"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(path), "-lm"], check=True)
    saved_lib, saved_path = oracle._lib, oracle._LIB_PATH
    try:
        oracle._lib = None
        oracle._LIB_PATH = str(so)
        oracle.build = lambda force=False, _p=str(so): _p  # noqa: E731 -- load the mutant
        caught = 0
        for check in PIN_CHECKS:
            try:
                check()
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin caught mutation: {name}"
    finally:
        oracle._lib, oracle._LIB_PATH = saved_lib, saved_path
        import importlib
        importlib.reload(oracle)
