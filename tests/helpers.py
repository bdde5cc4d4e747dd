"""Shared assertions for the parity tests.

GEMM outputs are compared with the oracle's float64 product of the exactly dequantized
operands, D = A . B^T, on the same packed inputs, by two criteria:

* the stated tolerance for fp32 outputs: max|diff| <= 1e-3 max|ref| and relative
  Frobenius error <= 1e-4 over the compared block;
* a per-element budget for the fp32 accumulation. The tensor core sums the exact
  products of each scale block and adds the block sums into an fp32 accumulator, so an
  element's error is a sum of n ~ K/16 roundings, each at most u = 2^-24 of the running
  sum, which is bounded by S = sum_k |a_k b_k| (the oracle's |A| . |B|^T). The worst case
  is n u S; the probabilistic bound of Higham and Mary ("A New Approach to Probabilistic
  Rounding Error Analysis", SIAM J. Sci. Comput. 41(5), 2019, Theorem 2.4) is
  lambda sqrt(n) u S, failing with probability at most 2 exp(-lambda^2 / 2) (lambda = 16:
  < 1e-55). The budget is lambda sqrt(n) u S plus 2u |ref| for the output scaling. A wrong
  scale on any tile, or one block's products dropped, breaks it even where the output is
  small, which a tolerance relative to max|ref| over the whole matrix would not see.

bf16 outputs are the nearest-even bf16 of the fp32 result, so each must lie between the
nearest-even bf16 of ref - budget and of ref + budget (rounding is monotone): at most one
bf16 ulp from the rounded reference, and only where the reference lies within the budget
of a rounding boundary.
"""
import math

import numpy as np

# stated tolerance for the fp32-output GEMMs
GEMM_MAXDIFF_REL = 1e-3
GEMM_FRO_REL = 1e-4
# per-element accumulation budget (module docstring)
U_FP32 = 2.0 ** -24
LAMBDA = 16.0


def assert_bytes_equal(got, ref, what):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    bad = got != ref
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ", ".join(f"{tuple(i)}: {got[tuple(i)]:#04x} vs {ref[tuple(i)]:#04x}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first {detail}")


def _split(ref):
    if isinstance(ref, tuple) and len(ref) == 3:
        d, s, k = ref
        return np.asarray(d, dtype=np.float64), np.asarray(s, dtype=np.float64), int(k)
    raise TypeError("GEMM references are (D, |A||B|^T, K): call the oracle with with_abs=True")


def ref_rows(ref, sl):
    """The rows `sl` of an oracle GEMM reference (D, |A||B|^T, K)."""
    d, s, k = ref
    return d[sl], s[sl], k


def accumulation_budget(ref, abs_prod, K):
    """Per-element error budget of an fp32-accumulated block-scaled product (docstring)."""
    n = max(1, K // 16)
    return LAMBDA * math.sqrt(n) * U_FP32 * abs_prod + 2 * U_FP32 * np.abs(ref)


def assert_gemm_close(got, ref, what):
    """fp32 GEMM output against the oracle reference (D, |A||B|^T, K)."""
    d, s, K = _split(ref)
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == d.shape, f"{what}: shape {got.shape} vs {d.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - d)
    md = np.max(err)
    mref = np.max(np.abs(d))
    fro = np.linalg.norm(got - d) / max(np.linalg.norm(d), 1e-300)
    assert md <= GEMM_MAXDIFF_REL * mref and fro <= GEMM_FRO_REL, (
        f"{what}: max|diff| {md:.3e} vs max|ref| {mref:.3e}, relative Frobenius {fro:.3e}")
    budget = accumulation_budget(d, s, K)
    bad = err > budget
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond the accumulation budget; "
                             f"first {i}: got {got[i]!r} ref {d[i]!r} sum|ab| {s[i]!r}")


def bf16_values(u16):
    """uint16 bf16 bit patterns -> float32 values."""
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32)


def round_to_bf16(x):
    """float64 -> nearest-even bf16 value (as float64), straight from float64 (no detour
    through fp32, which could round twice). Finite inputs in bf16's normal and subnormal
    range; bf16 keeps 8 significant bits and its smallest spacing is 2^-133."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # subnormal range: fixed spacing 2^-133
    q = np.rint(np.ldexp(x, 8 - e))          # round half to even on the bf16 grid
    return np.ldexp(q, e - 8)


def assert_bf16_rounding_of(got_bf16_u16, ref, what):
    """bf16 GEMM output: got lies in [bf16(ref - budget), bf16(ref + budget)]."""
    d, s, K = _split(ref)
    got = bf16_values(got_bf16_u16).astype(np.float64)
    assert got.shape == d.shape, f"{what}: shape {got.shape} vs {d.shape}"
    budget = accumulation_budget(d, s, K)
    lo, hi = round_to_bf16(d - budget), round_to_bf16(d + budget)
    bad = (got < lo) | (got > hi)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} bf16 outputs outside the rounding of "
                             f"ref +- budget; first {i}: got {got[i]!r} ref {d[i]!r} allowed [{lo[i]!r}, {hi[i]!r}]")


def assert_bf16_near(got_u16, want64, ulps, what):
    """bf16 results within `ulps` bf16 ulps of a float64 value (the epilogue's GELU is not
    correctly rounded, so the last bf16 bit may differ)."""
    got = bf16_values(got_u16).astype(np.float64)
    want = np.asarray(want64, dtype=np.float64)
    tol = ulps * np.maximum(np.abs(want), 2.0 ** -126) * 2.0 ** -7 + 2.0 ** -133
    bad = np.abs(got - want) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond {ulps} bf16 ulp; first "
                           f"got {got[bad][0]!r} want {want[bad][0]!r}")
