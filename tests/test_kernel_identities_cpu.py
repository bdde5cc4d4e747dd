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
