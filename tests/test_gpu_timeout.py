"""Failure detection on the GPU without a fault: the GEMM's bounded waits.

Every mbarrier wait of the CTA-pair GEMM gives up after a limit, raises the library's
device error word and ends its role, so a pipeline that never completes (a lost copy, a
peer that never arrives) returns an error status instead of hanging the GPU. The test
entry point launches the real kernel with its producers issuing no copies and a 20 ms
limit: every wait runs out, fp4q_device_status reports FP4Q_ERR_TIMEOUT, nothing was
written, and the context stays usable for the next (normal) GEMM."""
import time

import numpy as np
import pytest
import torch

from helpers import assert_gemm_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def rand_mxfp8(rng, rows, k):
    c = rng.integers(0, 0x7F, (rows, k), dtype=np.uint8) | (rng.integers(0, 2, (rows, k), dtype=np.uint8) << 7)
    return c, rng.integers(120, 135, (rows, k // 32), dtype=np.uint8)


def test_bounded_waits_run_out_and_report_timeout(F, orc):
    M, N, K = 512, 512, 1024
    rng = np.random.default_rng(3)
    a, asc = rand_mxfp8(rng, M, K)
    b, bsc = rand_mxfp8(rng, N, K)
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    ad, asd, bd, bsd = cu(a), cu(asc), cu(b), cu(bsc)
    d = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    assert F.fp4q_device_status() == F.OK
    for _ in range(2):
        t0 = time.perf_counter()
        assert F.fp4q_test_gemm_wait_timeout(ad, asd, bd, bsd, d, M, N, K, 20_000_000) == F.OK
        assert F.fp4q_device_status() == F.ERR_TIMEOUT
        assert time.perf_counter() - t0 < 10.0
        assert F.fp4q_device_status() == F.OK          # the word was cleared
        assert bool(torch.all(d == 7.0))               # the epilogue never ran
    # the context is intact: the same GEMM now runs normally and matches the oracle
    out = F.gemm_mxfp8(ad, asd, bd, bsd, torch.float32)
    assert F.fp4q_device_status() == F.OK
    assert_gemm_close(out.cpu().numpy(), orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), "GEMM after the timeout")
