"""The per-token activation form (4bit.vizuara.ai §10: one FP32 outer scale per row, Four Over
Six block scales) against the oracle: fp4q_quantize_1d_rows bit for bit (codes, scales and
per-row s_dec) on ragged, padded, long and degenerate rows and on sampled rows of the full-size
activations; fp4q_gemm_nvfp4_rows and fp4q_gemm_nvfp4_gelu_rows within the GEMM tolerance; the
requantize input kind FP4Q_IN_NVFP4_1D_ROWS bit for bit in every mode."""
import numpy as np
import pytest
import torch

from helpers import (assert_bf16_near, assert_bf16_rounding_of, assert_bytes_equal, assert_gemm_close,
                     bf16_values)
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check_rows(F, orc, x, four_six, what, ld_pad=0):
    rows, cols = x.shape
    if ld_pad:
        buf = torch.zeros(rows, cols + ld_pad, dtype=torch.bfloat16)
        buf[:, :cols] = x
        xd = buf.cuda()[:, :cols]
    else:
        xd = x.cuda()
    codes, scales, sd = F.quantize_1d_rows(xd, four_six)
    torch.cuda.synchronize()
    oc, os_, osd = orc.quantize_1d_rows(I.bf16_bits(x), four_six)
    assert_bytes_equal(scales.cpu().numpy(), os_, what + " scales")
    assert_bytes_equal(codes.cpu().numpy(), oc, what + " codes")
    assert np.array_equal(sd.cpu().numpy().view(np.uint32), osd.view(np.uint32)), what + " s_dec"
    return codes, scales, sd


# ------------------------------------------------------------------ quantize
@pytest.mark.parametrize("four_six", [False, True])
@pytest.mark.parametrize("rows,cols", [(256, 512), (1, 16), (3, 48), (17, 272), (9, 4096 + 16),
                                       (5, 16384), (3, 20480 + 32)])
def test_quantize_rows_shapes(F, orc, rows, cols, four_six):
    """One warp per row up to eight, rows held in registers up to 16384 values, and the
    re-read path of longer rows."""
    check_rows(F, orc, I.normal_with_outliers(rows, cols, seed=rows * 5 + cols), four_six,
               f"rows {rows}x{cols} 4/6={four_six}")


@pytest.mark.parametrize("four_six", [False, True])
def test_quantize_rows_padded_leading_dimension(F, orc, four_six):
    check_rows(F, orc, I.normal(40, 96, seed=3), four_six, "rows 40x96 ld+24", ld_pad=24)


def test_quantize_rows_degenerate_and_tie_rows(F, orc):
    x = torch.zeros(12, 64, dtype=torch.float32)
    x[1, 0] = 1e-30                                   # a lone tiny value: its row max
    x[2, :] = torch.linspace(-1, 1, 64)
    x[3, 16:32] = 1e-39                               # bf16 subnormals under a large row max
    x[3, 0] = 3e4
    x[4, :16] = 5.0                                   # equal values: both candidates exact
    x[5, 0], x[5, 16], x[5, 17] = 2688.0, 10.0, 7.5   # the 4 scale is exact, the 6 scale is not
    x[6, :] = -x[2, :]
    x[7, :32] = torch.tensor([6.0, 5.0, 4.0, 3.0] * 8)
    x[8, :] = 65280.0                                 # bf16 values near the top of the range
    x[9, :] = torch.arange(64) % 7 - 3.0
    x[10, ::2] = 1.0
    check_rows(F, orc, x.to(torch.bfloat16), True, "degenerate 4/6")
    check_rows(F, orc, x.to(torch.bfloat16), False, "degenerate")


def test_quantize_rows_gelu_output_distribution(F, orc):
    """The second layer's input: GELU of a Gaussian (one-sided, many small values)."""
    h = I.normal(64, 4096, seed=41)
    check_rows(F, orc, torch.nn.functional.gelu(h.float()).to(torch.bfloat16), True, "GELU(h) 64x4096")


def test_quantize_rows_full_size_sampled(F, orc):
    """The MLP's activations at full size (tokens 16384: X [16384, 4096] and GELU(h)
    [16384, 16384]); rows are independent, so sampled rows are checked against the oracle."""
    rng = np.random.default_rng(5)
    for shape, seed in (((16384, 4096), 51), ((16384, 16384), 52)):
        x = I.normal_with_outliers(*shape, seed=seed)
        codes, scales, sd = F.quantize_1d_rows(x.cuda(), True)
        torch.cuda.synchronize()
        pick = np.concatenate([[0, 1, shape[0] - 1], rng.choice(shape[0], 13, replace=False)])
        xs = I.bf16_bits(x[torch.from_numpy(pick)])
        oc, os_, osd = orc.quantize_1d_rows(xs, True)
        assert_bytes_equal(scales.cpu().numpy()[pick], os_, f"{shape} scales")
        assert_bytes_equal(codes.cpu().numpy()[pick], oc, f"{shape} codes")
        assert np.array_equal(sd.cpu().numpy()[pick], osd)
        del x, codes, scales, sd


# ------------------------------------------------------------------ GEMM with per-row outer scales
def rand_nvfp4(rng, rows, k, two_d=False):
    codes = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    shape = (rows // 16, k // 16) if two_d else (rows, k // 16)
    return codes, rng.integers(0x18, 0x58, shape, dtype=np.uint8)


@pytest.mark.parametrize("M,N,K,two_d", [(128, 256, 256, False), (300, 272, 768, True), (512, 512, 4096, True),
                                          (1, 16, 256, True), (96, 48, 512, False)])
def test_gemm_nvfp4_rows(F, orc, M, N, K, two_d):
    """Both the single-CTA kernel (M <= 128) and the CTA-pair kernel."""
    rng = np.random.default_rng(M * 3 + N + K)
    a, asc = rand_nvfp4(rng, M, K)
    b, bsc = rand_nvfp4(rng, N, K, two_d)
    asd = rng.uniform(0.05, 4.0, M).astype(np.float32)
    bsd = float(np.float32(1 / 3))
    kind = 2 if two_d else 1
    d = F.gemm_nvfp4_rows(cu(a), cu(asc), cu(asd), cu(b), cu(bsc), kind,
                          torch.tensor([bsd], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert_gemm_close(d.cpu().numpy(), orc.gemm_nvfp4_rows(a, asc, asd, b, bsc, kind, bsd, with_abs=True),
                      f"NVFP4 rows {M}x{N}x{K}")


@pytest.mark.parametrize("K", [512, 1024])
def test_gemm_nvfp4_rows_grouped(F, orc, K):
    """K = 512: the single-CTA kernel; K = 1024: the grouped CTA-pair kernel."""
    rng = np.random.default_rng(9 + K)
    G, N = 3, 64
    offs = [0, 100, 100, 260]
    M = offs[-1]
    a, asc = rand_nvfp4(rng, M, K)
    asd = rng.uniform(0.1, 2.0, M).astype(np.float32)
    bs = [rand_nvfp4(rng, N, K, True) for _ in range(G)]
    bsd = np.array([0.5, 0.25, 2.0], np.float32)
    d = F.gemm_nvfp4_rows(cu(a), cu(asc), cu(asd), cu(np.stack([c for c, _ in bs])),
                          cu(np.stack([s for _, s in bs])), F.SCALE_2D, cu(bsd), torch.float32, G, offs)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    got = d.cpu().numpy()
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        ref = orc.gemm_nvfp4_rows(a[lo:hi], asc[lo:hi], asd[lo:hi], bs[g][0], bs[g][1], 2, float(bsd[g]), with_abs=True)
        assert_gemm_close(got[lo:hi], ref, f"group {g}")


@pytest.mark.parametrize("M,N,K", [(300, 272, 4096), (96, 256, 512)])
def test_gemm_nvfp4_gelu_rows(F, orc, M, N, K):
    """h equals the plain per-row GEMM's bf16 output bit for bit and is within one bf16 ulp of
    the oracle; act = GELU(h) within one bf16 ulp of float64 GELU of those bf16 values."""
    x = I.normal_with_outliers(M, K, seed=M + 7)
    w = I.normal(N, K, seed=N + 8, std=0.02)
    xc, xs, xsd = F.quantize_1d_rows(x.cuda(), True)
    wc, ws, wsd, _ = F.quantize_2d(w.cuda())
    h, act = F.gemm_nvfp4_gelu_rows(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd)
    plain = F.gemm_nvfp4_rows(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert np.array_equal(u16(h), u16(plain))
    ref = orc.gemm_nvfp4_rows(xc.cpu().numpy(), xs.cpu().numpy(), xsd.cpu().numpy(),
                              wc.cpu().numpy(), ws.cpu().numpy(), 2, float(wsd.item()), with_abs=True)
    assert_bf16_rounding_of(u16(h), ref, f"GELU rows GEMM h {M}x{N}x{K}")
    assert_bf16_near(u16(act), orc.gelu_bf16(u16(h)), 1, f"GELU(h) rows {M}x{N}x{K}")


# ------------------------------------------------------------------ requantize from per-row input
CASES = [(t, r, m) for t in (0, 1) for r in (0, 1) for m in (0, 1)]


@pytest.mark.parametrize("transpose,rht,rounding", CASES)
def test_requant_rows_input_all_modes(F, orc, transpose, rht, rounding):
    rows, cols = 96, 160
    seed, signs, tag = 0x0BAD_5EED_1234_5678, 0x5AC3, 4
    x = I.normal_with_outliers(rows, cols, seed=61)
    oc, os_, osd = orc.quantize_1d_rows(I.bf16_bits(x), True)
    e4, e8 = F.requant_mxfp8(F.IN_NVFP4_1D_ROWS, cu(oc), cu(os_), cu(osd), rows, cols, transpose, rht, signs,
                             rounding, seed, tag)
    torch.cuda.synchronize()
    r4, r8 = orc.requant_mxfp8(orc.IN_NVFP4_1D_ROWS, oc, os_, osd, rows, cols, transpose, rht, signs,
                               rounding, seed, tag)
    what = f"rows-input T={transpose} rht={rht} sr={rounding}"
    assert_bytes_equal(e8.cpu().numpy(), r8, what + " e8m0")
    assert_bytes_equal(e4.cpu().numpy(), r4, what + " e4m3")


def test_requant_rows_input_wgrad_full_size_sampled(F, orc):
    """X_q^T with per-row outer scales at the MLP's size (tokens 16384 x 4096), RHT + SR."""
    M, K = 16384, 4096
    seed, signs = I.sr_seed(6), I.rht_signs(6)
    x = I.normal_with_outliers(M, K, seed=62)
    xc, xs, xsd = F.quantize_1d_rows(x.cuda(), True)
    e4, e8 = F.requant_mxfp8(F.IN_NVFP4_1D_ROWS, xc, xs, xsd, M, K, 1, 1, signs, F.SR, seed, F.TAG_XT)
    torch.cuda.synchronize()
    oc, os_, osd = xc.cpu().numpy(), xs.cpu().numpy(), xsd.cpu().numpy()
    e4, e8 = e4.cpu().numpy(), e8.cpu().numpy()
    for r in (0, 1, 2047, 4095):
        r4, r8 = orc.requant_mxfp8(orc.IN_NVFP4_1D_ROWS, oc, os_, osd, M, K, 1, 1, signs, orc.SR, seed,
                                   F.TAG_XT, out_rows=(r, r + 1))
        assert_bytes_equal(e8[r:r + 1], r8, f"X_q^T e8m0 row {r}")
        assert_bytes_equal(e4[r:r + 1], r4, f"X_q^T e4m3 row {r}")


# ------------------------------------------------------------------ the layer
def test_linear_layer_with_per_token_activations(F, orc):
    """linear_forward(outer="row") quantizes x per token with 4/6 and multiplies with the
    per-row GEMM; its backward requantizes X_q from the per-row form."""
    from mxfp8_precision_numerics_gb300 import layer
    M, K, N = 256, 512, 256
    x = I.normal_with_outliers(M, K, seed=71)
    w = I.normal(N, K, seed=72, std=0.02)
    y, saved = layer.linear_forward(x.cuda(), w.cuda(), out_dtype=torch.float32, outer="row")
    dy = I.student_t(M, N, seed=73)
    dx, dw = layer.linear_backward(dy.cuda(), saved, I.sr_seed(7), I.rht_signs(7))
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    oc, os_, osd = orc.quantize_1d_rows(I.bf16_bits(x), True)
    assert_bytes_equal(saved.xq[0].cpu().numpy(), oc, "layer x codes")
    wc, ws, _, wsd = orc.quantize_2d(I.bf16_bits(w))
    assert_gemm_close(y.cpu().numpy(), orc.gemm_nvfp4_rows(oc, os_, osd, wc, ws, 2, wsd, with_abs=True), "layer y")
    ref = (x.float() @ w.float().t()).numpy()
    assert np.linalg.norm(y.cpu().numpy() - ref) / np.linalg.norm(ref) < 0.15
    assert dx.shape == (M, K) and dw.shape == (N, K)
    assert torch.isfinite(dx.float()).all() and torch.isfinite(dw).all()


def test_readme_example_runs(F):
    """The usage example of the repository's front page, as written there."""
    from mxfp8_precision_numerics_gb300 import layer
    x = torch.randn(4096, 4096, device="cuda").to(torch.bfloat16)
    w = (0.02 * torch.randn(4096, 4096, device="cuda")).to(torch.bfloat16)
    y, saved = layer.linear_forward(x, w, out_dtype=torch.bfloat16, outer="row")
    dy = torch.randn_like(y)
    dx, dw = layer.linear_backward(dy, saved, seed=1234, rht_signs=0xA5C3)
    codes, scales, s_dec, amax = F.quantize_1d(x)
    wc, wt, ws_dec, _ = F.quantize_2d(w)
    d = F.gemm_nvfp4(codes, scales, s_dec, wc, wt, F.SCALE_2D, ws_dec, torch.float32)
    assert F.fp4q_device_status() == F.OK
    ref = x.float() @ w.float().t()
    assert float((d - ref).norm() / ref.norm()) < 0.15 and float((y.float() - ref).norm() / ref.norm()) < 0.15
    assert dx.shape == x.shape and dw.shape == w.shape
