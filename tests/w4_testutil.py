"""Helpers shared by the GPU parity tests: device upload and the comparison
rules.  The rules follow the library's stated tolerances:
  * relative L2 error of the fp32 output (before the bfloat16 cast) <= 1e-3,
  * max |error| <= 1e-2 * max |y_ref|,
  * bfloat16 output within 1 ulp of round-to-nearest-even(y_ref) -- except
    where a bfloat16 ulp at y_ref is smaller than the fp32 rounding-error bound
    of the sum itself (tiny |y_ref| from cancellation), in which case the fp32
    output must lie within that bound, |y_ref| must be at most 2^9 times the
    bound, and such outputs must be at most 1 % of the comparison.
The bound is the textbook one for a sum evaluated with n sequential roundings,
|error| <= n * u * A, with u = 2^-23 (one fp32 ulp, which also covers
truncating accumulation), n = 8 k-steps per group + G groups + the number of K
splits + 1, and A the sum of the magnitudes of the terms that are actually
rounded:
  * exact zero-point subtraction (A = q - z in the tensor-core operand, the
    workspace split): A = sum_k |w_k x_k| (the oracle's `with_abs` sum);
  * zero point folded out of the inner product (the cluster split, fp16
    operands: per group d0 = sum over S01 of (1024 + q) x and d1 / 16 = sum
    over S23 of (64 + q) x, minus (1024 + z) X01 and (64 + z) X23, where
    S01 = {k : k mod 16 < 8}, S23 the rest, X the sums of x over them):
    A = folded_abs(), and n grows by 8 for the group sums (a tree of at most
    7 levels, then the fma).  x enters as fp16 scaled per token by a power of
    two into [2^14, 2^15): exact except for values more than 2^28 below the
    token's largest, whose rounding (at most 2^-39 times that largest value
    each) the bound also covers.
"""
from __future__ import annotations

import numpy as np

import oracle

REL_L2 = 1e-3
MAX_ABS_FRAC = 1e-2
# Outputs more than one bf16 ulp from RNE(y_ref) (allowed only inside the fp32
# bound): at most this fraction of a comparison, each with |y_ref| at most
# this multiple of its bound (2^9: one bf16 ulp is at least 2^-8 |y|, with a
# factor 2 for the rounding of the larger of the two values).
OFF_ULP_MAX_FRACTION = 0.01
OFF_ULP_MAX_REF_OVER_BOUND = 2.0 ** 9
# (what, outputs off by more than one ulp, outputs compared) of every
# check_gemv call in the session; summarised at the end of the test run.
OFF_ULP_STATS = []


def to_device(p, dev="cuda"):
    import torch
    qw = torch.from_numpy(np.ascontiguousarray(p.qweight).view(np.int32)).to(dev)
    sc = torch.from_numpy(np.ascontiguousarray(p.scales).view(np.int16)).to(dev)
    zp = torch.from_numpy(np.ascontiguousarray(p.zeros)).to(dev)
    x = torch.from_numpy(np.ascontiguousarray(p.x).view(np.int16)).to(dev).view(torch.bfloat16)
    return qw, sc, zp, x


def x_to_device(xbits, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(xbits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map bfloat16 bit patterns to integers whose difference counts ulps."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


FOLD_EXTRA_STEPS = 8


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def folded_abs(p, rows=None) -> np.ndarray:
    """Per output [M, len(rows)]: sum over groups g of |s_g| * (sum_{S01} (1024 + q)|x|
    + sum_{S23} (64 + q)|x| + (1024 + z) sum_{S01} |x| + (64 + z) sum_{S23} |x|),
    the magnitudes rounded by the folded arithmetic, plus the fp16 rounding of
    tiny x, in units of the bound's u = 2^-23.  The tensor-core product sees
    the fp16 value x16 and the zero-point term the fp32 sum of the scaled x,
    so each weight adds |s| (1024 + q or 64 + q) |x16 - x|: at most half an
    fp16 subnormal step, 2^-25, over the token's scale 2^e, which is at most
    2^-39 max |x| (2^e max |x| >= 2^14), or 2^-151 where e is clamped."""
    rows = np.arange(p.N) if rows is None else np.asarray(rows)
    K, M = p.K, p.M
    G = K // 128
    words = np.asarray(p.qweight)[rows].astype(np.uint32)
    q = np.empty((len(rows), K), np.float64)
    for j in range(8):
        q[:, j::8] = (words >> np.uint32(4 * j)) & np.uint32(0xF)
    s = np.abs(np.asarray(p.scales)[rows].view(np.float16).astype(np.float64))   # [R, G]
    z = np.asarray(p.zeros)[rows].astype(np.float64)                              # [R, G]
    xa = np.abs(_bf16_to_f64(p.x)).reshape(M, G, 128)                             # [M, G, 128]
    lo = (np.arange(128) % 16) < 8                                                # S01
    a = np.where(lo[None, None, :], 1024.0, 64.0) + q.reshape(len(rows), G, 128)
    out = np.empty((M, len(rows)))
    for m in range(M):
        t = np.einsum("rgk,gk->rg", a, xa[m]) + (1024.0 + z) * xa[m][:, lo].sum(-1)[None, :] \
            + (64.0 + z) * xa[m][:, ~lo].sum(-1)[None, :]
        tiny = (a * s[:, :, None]).sum((1, 2)) * max(xa[m].max() * 2.0 ** -39, 2.0 ** -151) \
            / 2.0 ** -23
        out[m] = (s * t).sum(-1) + tiny
    return out


def check_gemv(got32: np.ndarray, got16: np.ndarray, ref64: np.ndarray, refabs: np.ndarray,
               K: int, splits: int, what: str = "", extra_steps: int = 0) -> dict:
    ref32 = ref64.astype(np.float32)
    err = got32.astype(np.float64) - ref64
    nref = np.linalg.norm(ref32.astype(np.float64))
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    maxabs = np.abs(err).max() if err.size else 0.0
    maxref = np.abs(ref32).max() if ref32.size else 0.0
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    assert maxabs <= MAX_ABS_FRAC * maxref + 0.0, f"{what}: max abs error {maxabs:.3e}"
    want16 = oracle.bf16_rne(ref32)
    ulps = np.abs(ordered(got16) - ordered(want16))
    off = ulps > 1
    n_steps = 8 + K // 128 + splits + 1 + extra_steps
    bound = n_steps * 2.0 ** -23 * refabs
    if off.any():
        worst = np.abs(err[off]) - bound[off]
        assert (worst <= 0).all(), (
            f"{what}: {int(off.sum())} bf16 outputs off by >1 ulp beyond the fp32 bound "
            f"(worst excess {worst.max():.3e})")
        # Two bf16 roundings can end more than one ulp apart only if the fp32
        # values differ by at least one bf16 ulp, which is at least 2^-8 of
        # the smaller magnitude: so every such element has |y_ref| within a
        # small multiple of its fp32 bound (cancellation), never an ordinary one.
        assert (np.abs(ref64[off]) <= OFF_ULP_MAX_REF_OVER_BOUND * bound[off]).all(), (
            f"{what}: an output off by >1 ulp has |y_ref| above "
            f"{OFF_ULP_MAX_REF_OVER_BOUND} x its fp32 bound")
    assert off.sum() <= OFF_ULP_MAX_FRACTION * off.size, (
        f"{what}: {int(off.sum())} of {off.size} bf16 outputs off by more than one ulp")
    # the bfloat16 output is the nearest-even rounding of the fp32 output
    assert np.array_equal(got16, oracle.bf16_rne(got32)), f"{what}: bf16 != rne(fp32)"
    OFF_ULP_STATS.append((what, int(off.sum()), int(off.size)))
    return {"rel_l2": float(rel), "max_abs": float(maxabs), "ulp_gt1": int(off.sum())}
