"""fp4q_quantize_2d_noalloc — the weight quantizer for callers that cannot allocate device
memory (its amax workspace is a fixed array inside the library) — must give exactly the
bytes of fp4q_quantize_2d. Two calls in a row check that the shared array is cleared between
calls: the first batch has a far larger amax than the second, so a stale maximum would change
the second call's scales. This file sorts last so a stop-at-first-failure run has already run
every other test."""
import ctypes

import pytest
import torch

from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def _both(F, w):
    """-> (codes, tiles, s_dec) from the allocating and the allocation-free entry points."""
    batch, rows, cols = w.shape
    ref = F.quantize_2d(w)
    codes = torch.empty((batch, rows, cols // 2), dtype=torch.uint8, device="cuda")
    tiles = torch.empty((batch, rows // 16, cols // 16), dtype=torch.uint8, device="cuda")
    s_dec = torch.empty((batch,), dtype=torch.float32, device="cuda")
    F.fp4q_quantize_2d_noalloc(w, rows, cols, w.stride(1), batch, w.stride(0), codes, tiles, s_dec)
    torch.cuda.synchronize()
    return ref[:3], (codes, tiles, s_dec)


def test_noalloc_quantize_2d_matches_two_calls_in_a_row(F):
    big = torch.stack([I.normal_with_outliers(64, 272, seed=70 + e, std=1.0) for e in range(3)]).cuda()
    small = torch.stack([I.normal(64, 272, seed=80 + e, std=0.02) for e in range(3)]).cuda()
    for w in (big, small):
        (rc, rt, rd), (c, t, d) = _both(F, w)
        assert torch.equal(c, rc) and torch.equal(t, rt)
        assert torch.equal(d, rd)


def test_noalloc_rejects_a_batch_beyond_the_fixed_array(F):
    w = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(16 * 8, dtype=torch.uint8, device="cuda")
    st = F._lib.fp4q_quantize_2d_noalloc(ctypes.c_void_p(w.data_ptr()), 16, 16, 16,
                                         F.NOALLOC_MAX_BATCH + 1, 256, ctypes.c_void_p(out.data_ptr()),
                                         ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         None)
    assert st == F.ERR_SHAPE
