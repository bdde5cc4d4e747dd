"""Arithmetic identities the CUDA kernels rely on, checked exhaustively on the host.

These do not touch the GPU: each shows that a cheaper evaluation used inside a kernel gives,
for every input the kernel can see, the same fp32 result as the operation the oracle states.
"""
from fractions import Fraction

import numpy as np


def rn32(fr):
    """Nearest float32 to the rational fr, ties to the even significand."""
    f = np.float32(float(fr))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - fr)
        if best is None or d < best[0] or (d == best[0] and (int(cand.view(np.uint32)) & 1) == 0):
            best = (d, cand)
    return np.float32(best[1])


def test_division_by_six_with_one_correction_step():
    """Block scales divide a block max (a bf16 value) by 6. The kernels compute
    q0 = a * RN(1/6), r = fma(-q0, 6, a), q = fma(r, RN(1/6), q0) (division by a constant
    with a correction step, Brisebarre, Muller and Raina, IEEE TC 2004); q equals the IEEE
    quotient RN(a / 6) for every non-negative finite bf16 a, subnormals included."""
    a_all = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    c = np.float32(1.0) / np.float32(6.0)
    assert c.view(np.uint32) == 0x3E2AAAAB
    C = Fraction(float(c))
    for a in a_all:
        A = Fraction(float(a))
        q0 = rn32(A * C)
        r = rn32(A - Fraction(float(q0)) * 6)
        q = rn32(Fraction(float(q0)) + Fraction(float(r)) * C)
        assert q.view(np.uint32) == rn32(A / 6).view(np.uint32), float(a)


def test_s2f6_code_by_magic_addition():
    """S2F6 encoding rounds t = y 2^(6-e) half to even and clamps it to [-128, 127]. The
    kernels clamp t first, add 1.5 * 2^23 in fp32 and keep the low byte of the sum's bits;
    that byte is the two's-complement code for every float32 t (checked on every float32
    in [-160, 160] whose significand ends in ten zero bits, on all halves and quarters of that
    range, and at the extremes)."""
    base = (np.arange(0, 1 << 22, dtype=np.uint32) << 10).view(np.float32)
    base = base[np.isfinite(base) & (np.abs(base) <= 160)]
    grid = np.arange(-160 * 4, 160 * 4 + 1, dtype=np.float32) / np.float32(4)
    extra = np.array([3.4e38, -3.4e38, 1e-45, -1e-45, 0.0, -0.0, 127.49999, 127.5, -128.5, -128.49998],
                     dtype=np.float32)
    t = np.concatenate([base, -base, grid, extra]).astype(np.float32)
    clamped = np.minimum(np.maximum(t, np.float32(-128)), np.float32(127))
    s = (clamped + np.float32(12582912.0)).astype(np.float32)      # one fp32 rounding (RNE)
    got = (s.view(np.uint32) & 0xFF).astype(np.uint8)
    want = np.clip(np.rint(t.astype(np.float64)), -128, 127).astype(np.int64).astype(np.int8).view(np.uint8)
    assert np.array_equal(got, want)


def test_s2f6_decode_by_biased_byte():
    """Decoding takes code c as the float with bits 0x4B000000 | (c + 128) (that is
    2^23 + c + 128), subtracts 2^23 + 128 and multiplies by the power-of-two step; both
    steps are exact, so the value is c * step for all 256 codes and every step the E8M0
    byte can give."""
    c = np.arange(256, dtype=np.uint32)
    f = (np.uint32(0x4B000000) | (c ^ np.uint32(0x80))).view(np.float32)
    q = (f - np.float32(8388736.0)).astype(np.float32)
    assert np.array_equal(q, c.astype(np.uint8).view(np.int8).astype(np.float32))
    for sc in range(0, 255):
        step = np.float32(np.ldexp(1.0, sc - 127 - 6))
        with np.errstate(over="ignore"):           # -128 * 2^121 is -inf on both sides
            got = (q * step).astype(np.float32)
            want = np.ldexp(c.astype(np.uint8).view(np.int8).astype(np.float64), sc - 133).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), sc
