"""Shared assertions for the parity tests."""
import math

import numpy as np

_erfc = np.vectorize(math.erfc)

# GEMM tolerance stated for the fp32-output GEMMs: max|diff| <= 1e-3 max|ref|, relative
# Frobenius error <= 1e-4, against the float64 product of the exactly dequantized operands.
GEMM_MAXDIFF_REL = 1e-3
GEMM_FRO_REL = 1e-4


def assert_bytes_equal(got, ref, what):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    bad = got != ref
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ", ".join(f"{tuple(i)}: {got[tuple(i)]:#04x} vs {ref[tuple(i)]:#04x}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first {detail}")


def assert_gemm_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    md = np.max(np.abs(got - ref))
    mref = np.max(np.abs(ref))
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert md <= GEMM_MAXDIFF_REL * mref and fro <= GEMM_FRO_REL, (
        f"{what}: max|diff| {md:.3e} vs max|ref| {mref:.3e}, relative Frobenius {fro:.3e}")


def bf16_values(u16):
    """uint16 bf16 bit patterns -> float32 values."""
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32)


def assert_bf16_rounding_of(got_bf16_u16, ref, what):
    """A bf16 GEMM output must be within one bf16 ulp of the nearest-even bf16 of the
    reference (the fp32 accumulation itself is within the GEMM tolerance)."""
    import oracle
    got = bf16_values(got_bf16_u16).astype(np.float64)
    ref32 = np.asarray(ref, dtype=np.float32)
    want = oracle.round_bf16(ref32).astype(np.float64)
    ulp = np.abs(want) * 2.0 ** -7 + 1e-30
    err = np.abs(got - want)
    tol = np.maximum(ulp, GEMM_MAXDIFF_REL * np.max(np.abs(ref)))
    bad = err > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} bf16 outputs off by more than one ulp"


def phi64(x):
    """Standard normal cdf as erfc(-x/sqrt 2)/2: no cancellation in the negative tail."""
    return 0.5 * _erfc(-np.asarray(x, dtype=np.float64) / math.sqrt(2.0))


def gelu64(x):
    x = np.asarray(x, dtype=np.float64)
    return x * phi64(x)


def gelu_grad64(x):
    x = np.asarray(x, dtype=np.float64)
    return phi64(x) + x * np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def assert_bf16_near(got_u16, want64, ulps, what):
    """bf16 results within `ulps` bf16 ulps of a float64 value (the epilogue's GELU is not
    correctly rounded, so the last bf16 bit may differ)."""
    got = bf16_values(got_u16).astype(np.float64)
    want = np.asarray(want64, dtype=np.float64)
    tol = ulps * np.maximum(np.abs(want), 2.0 ** -126) * 2.0 ** -7 + 2.0 ** -133
    bad = np.abs(got - want) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond {ulps} bf16 ulp; first "
                           f"got {got[bad][0]!r} want {want[bad][0]!r}")
