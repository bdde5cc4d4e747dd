"""MXFP4 (the format the pages compare NVFP4 with) against the oracle: fp4q_quantize_mxfp4 bit
for bit (with and without the 32-point rotation; ragged, padded and degenerate rows), and
fp4q_gemm_mxfp4 on the tensor cores within the GEMM tolerance (fp32) or one bf16 ulp."""
import numpy as np
import pytest
import torch

from helpers import assert_bf16_rounding_of, assert_bytes_equal, assert_gemm_close
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SIGNS = 0x5EED_1234


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_q(F, orc, x, rht, what, ld_pad=0):
    rows, cols = x.shape
    if ld_pad:
        buf = torch.zeros(rows, cols + ld_pad, dtype=torch.bfloat16)
        buf[:, :cols] = x
        xd = buf.cuda()[:, :cols]
    else:
        xd = x.cuda()
    codes, e8 = F.quantize_mxfp4(xd, rht, SIGNS)
    torch.cuda.synchronize()
    oc, oe = orc.quantize_mxfp4(I.bf16_bits(x), rht, SIGNS)
    assert_bytes_equal(e8.cpu().numpy(), oe, what + " e8m0")
    assert_bytes_equal(codes.cpu().numpy(), oc, what + " codes")
    return codes, e8


@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("rows,cols", [(256, 512), (3, 96), (33, 4096 + 32), (1, 32), (64, 2048), (5, 1024)])
def test_quantize_mxfp4_shapes(F, orc, rows, cols, rht):
    check_q(F, orc, I.normal_with_outliers(rows, cols, seed=rows + cols), rht, f"mxfp4 {rows}x{cols} rht={rht}")


def test_quantize_mxfp4_padded_and_degenerate(F, orc):
    check_q(F, orc, I.normal(40, 96, seed=3), False, "padded", ld_pad=24)
    for rht in (False, True):                        # several warps per row, padded rows
        check_q(F, orc, I.normal_with_outliers(9, 1024, seed=4), rht, f"padded 1024 rht={rht}", ld_pad=40)
    x = torch.zeros(6, 1024, dtype=torch.float32)
    x[1, 0] = 22.0                                   # the worked example: scale 4, 22 -> 24
    x[2, :32] = 1e-39                                # subnormal block
    x[3, 0] = 3.015625                               # amax 3 + delta keeps 3 as its top code
    x[4, :] = 1.0e37                                 # near the top of the range (its rotation stays finite)
    x[5, :] = torch.linspace(-6, 6, 1024)
    for width in (64, 1024):                         # degenerate rows alone, and among many groups
        xs = x[:, :width].contiguous()
        for rht in (False, True):
            check_q(F, orc, xs.to(torch.bfloat16), rht, f"degenerate {width} rht={rht}")
    x[4, :] = 3.0e38                                 # without the rotation: the largest bf16 values
    for width in (64, 1024):
        check_q(F, orc, x[:, :width].contiguous().to(torch.bfloat16), False, f"near-max {width}")


def rand_mxfp4(rng, rows, k):
    return rng.integers(0, 256, (rows, k // 2), dtype=np.uint8), rng.integers(118, 136, (rows, k // 32), dtype=np.uint8)


def test_gemm_mxfp4_structured_scales(F, orc):
    """Every code 1.0; the scales vary by row, by column and by 32-block, so a wrong scale
    column, lane or byte pair in tensor memory changes the result."""
    M, N, K = 256, 512, 2048
    a = np.full((M, K // 2), 0x22, np.uint8)
    b = np.full((N, K // 2), 0x22, np.uint8)
    kb = np.arange(K // 32)
    ae = (124 + (np.arange(M)[:, None] % 5) + (kb[None, :] % 3)).astype(np.uint8)
    be = (125 + (np.arange(N)[:, None] % 3) + (kb[None, :] % 4)).astype(np.uint8)
    d = F.gemm_mxfp4(cu(a), cu(ae), cu(b), cu(be))
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert_gemm_close(d.cpu().numpy(), orc.gemm_mxfp4(a, ae, b, be, with_abs=True), "MXFP4 structured")


@pytest.mark.parametrize("M,N,K", [(256, 256, 2048), (300, 272, 4096), (128, 512, 2048), (1, 16, 2048)])
def test_gemm_mxfp4_random(F, orc, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a, ae = rand_mxfp4(rng, M, K)
    b, be = rand_mxfp4(rng, N, K)
    ref = orc.gemm_mxfp4(a, ae, b, be, with_abs=True)
    d = F.gemm_mxfp4(cu(a), cu(ae), cu(b), cu(be))
    db = F.gemm_mxfp4(cu(a), cu(ae), cu(b), cu(be), torch.bfloat16)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert_gemm_close(d.cpu().numpy(), ref, f"MXFP4 {M}x{N}x{K}")
    assert_bf16_rounding_of(db.cpu().view(torch.int16).numpy().view(np.uint16), ref, f"MXFP4 bf16 {M}x{N}x{K}")


def test_mxfp4_linear_layer(F, orc):
    """Quantize X and W to MXFP4 (W with the rotation on both operands cancels in X W^T: the
    same rotation along K on both sides), multiply on the tensor cores, compare with the oracle
    and with the bf16 product."""
    M, N, K = 512, 256, 2048
    x = I.normal_with_outliers(M, K, seed=81)
    w = I.normal(N, K, seed=82, std=0.02)
    for rht in (False, True):
        xc, xe = F.quantize_mxfp4(x.cuda(), rht, SIGNS)
        wc, we = F.quantize_mxfp4(w.cuda(), rht, SIGNS)
        y = F.gemm_mxfp4(xc, xe, wc, we)
        torch.cuda.synchronize()
        oxc, oxe = orc.quantize_mxfp4(I.bf16_bits(x), rht, SIGNS)
        owc, owe = orc.quantize_mxfp4(I.bf16_bits(w), rht, SIGNS)
        assert_gemm_close(y.cpu().numpy(), orc.gemm_mxfp4(oxc, oxe, owc, owe, with_abs=True), f"MXFP4 layer rht={rht}")
        ref = (x.float() @ w.float().t()).numpy()
        assert np.linalg.norm(y.cpu().numpy() - ref) / np.linalg.norm(ref) < 0.2


def test_mxfp4_format_comparison_full_size_sampled(F, orc):
    """The format comparison's shape (X 16384 x 4096 with outliers, W 14336 x 4096, bf16 GEMM
    output), in the calls the benchmark times: both quantizers checked bit for bit on sampled
    rows (rows are independent), the GEMM's sampled output rows against the oracle's product of
    the device's own codes (within one bf16 ulp), with and without the rotation."""
    M, K, N = 16384, 4096, 14336
    x = I.normal_with_outliers(M, K, seed=3)
    w = I.normal(N, K, seed=30, std=0.02)
    rows = np.sort(np.random.default_rng(1).choice(M, 32, replace=False))
    rows[0], rows[-1] = 0, M - 1
    wrows = np.sort(np.random.default_rng(2).choice(N, 32, replace=False))
    idx = torch.from_numpy(rows).cuda()
    for rht in (False, True):
        xc, xe = F.quantize_mxfp4(x.cuda(), rht, SIGNS)
        wc, we = F.quantize_mxfp4(w.cuda(), rht, SIGNS)
        y = F.gemm_mxfp4(xc, xe, wc, we, torch.bfloat16)
        torch.cuda.synchronize()
        assert F.fp4q_device_status() == F.OK
        oc, oe = orc.quantize_mxfp4(I.bf16_bits(x[rows]), rht, SIGNS)
        assert_bytes_equal(xc[idx].cpu().numpy(), oc, f"X codes rht={rht}")
        assert_bytes_equal(xe[idx].cpu().numpy(), oe, f"X e8m0 rht={rht}")
        oc, oe = orc.quantize_mxfp4(I.bf16_bits(w[wrows]), rht, SIGNS)
        widx = torch.from_numpy(wrows).cuda()
        assert_bytes_equal(wc[widx].cpu().numpy(), oc, f"W codes rht={rht}")
        assert_bytes_equal(we[widx].cpu().numpy(), oe, f"W e8m0 rht={rht}")
        ref = orc.gemm_mxfp4(xc[idx].cpu().numpy(), xe[idx].cpu().numpy(), wc.cpu().numpy(), we.cpu().numpy(), with_abs=True)
        yb = y[idx].cpu().view(torch.int16).numpy().view(np.uint16)
        assert_bf16_rounding_of(yb, ref, f"MXFP4 16384x14336x4096 sampled rht={rht}")
