"""The GEMMs with the MLP's activation fused into the epilogue (fp4q_gemm_nvfp4_gelu,
fp4q_gemm_mxfp8_dgelu): the GEMM part against the oracle's float64 product (one bf16 ulp,
as for every bf16 GEMM output) and bit-identical to the plain GEMM's bf16 output; the
activation part against GELU(x) = x Phi(x) and GELU'(x) = Phi(x) + x phi(x) evaluated in
float64 on the very bf16 values the epilogue started from; the |GELU| maximum exactly."""
import numpy as np
import pytest
import torch

from helpers import assert_bf16_near, assert_bf16_rounding_of, bf16_values
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(300, 272, 4096), (96, 256, 512), (512, 512, 1024)])
def test_nvfp4_gelu_epilogue(F, orc, M, N, K):
    x = I.normal_with_outliers(M, K, seed=M + 3)
    w = I.normal(N, K, seed=N + 4, std=0.02)
    xc, xs, xsd, _ = F.quantize_1d(x.cuda())
    wc, ws, wsd, _ = F.quantize_2d(w.cuda())
    h, act, amax = F.gemm_nvfp4_gelu(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd)
    plain = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    # h is the plain GEMM's bf16 output, bit for bit, and within one ulp of the oracle
    assert np.array_equal(u16(h), u16(plain)), "h differs from the plain GEMM output"
    ref = orc.gemm_nvfp4(xc.cpu().numpy(), xs.cpu().numpy(), 1, float(xsd.item()),
                         wc.cpu().numpy(), ws.cpu().numpy(), 2, float(wsd.item()), with_abs=True)
    assert_bf16_rounding_of(u16(h), ref, f"GELU GEMM h {M}x{N}x{K}")
    assert_bf16_near(u16(act), orc.gelu_bf16(u16(h)), 1, f"GELU(h) {M}x{N}x{K}")
    av = bf16_values(u16(act))
    assert float(amax.item()) == float(np.max(np.abs(av))), "amax is not max|GELU(h)|"


def test_nvfp4_gelu_amax_feeds_quantize(F):
    """quantize_1d(act, amax_in=act_amax) equals quantize_1d(act) computing its own amax."""
    x = I.normal_with_outliers(256, 512, seed=11)
    w = I.normal(512, 512, seed=12, std=0.02)
    xc, xs, xsd, _ = F.quantize_1d(x.cuda())
    wc, ws, wsd, _ = F.quantize_2d(w.cuda())
    _, act, amax = F.gemm_nvfp4_gelu(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd)
    c1, s1, d1, a1 = F.quantize_1d(act, amax_in=amax)
    c2, s2, d2, a2 = F.quantize_1d(act)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(s1, s2) and float(d1.item()) == float(d2.item())
    assert float(a1.item()) == float(a2.item())


def rand_mxfp8(rng, rows, k):
    c = rng.integers(0, 0x7F, (rows, k), dtype=np.uint8) | (rng.integers(0, 2, (rows, k), dtype=np.uint8) << 7)
    return c, rng.integers(118, 128, (rows, k // 32), dtype=np.uint8)


@pytest.mark.parametrize("M,N,K", [(300, 272, 4096), (96, 256, 512), (512, 512, 1024)])
def test_mxfp8_dgelu_epilogue(F, orc, M, N, K):
    rng = np.random.default_rng(M * 13 + N)
    a, asc = rand_mxfp8(rng, M, K)
    b, bsc = rand_mxfp8(rng, N, K)
    h = I.normal(M, N, seed=M + N, std=1.5)                   # a pre-activation in GELU's curved range
    cu = lambda t: torch.from_numpy(np.ascontiguousarray(t)).cuda()
    dh = F.gemm_mxfp8_dgelu(cu(a), cu(asc), cu(b), cu(bsc), h.cuda())
    da = F.gemm_mxfp8(cu(a), cu(asc), cu(b), cu(bsc), torch.bfloat16)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert_bf16_rounding_of(u16(da), orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), f"dgrad {M}x{N}x{K}")
    want = bf16_values(u16(da)).astype(np.float64) * orc.gelu_bf16(I.bf16_bits(h), grad=True)
    assert_bf16_near(u16(dh), want, 2, f"dGELU {M}x{N}x{K}")
