"""tcgen05 block-scaled GEMMs (fp4q_gemm_nvfp4 / fp4q_gemm_mxfp8) against the oracle's
float64 product of the exactly dequantized operands, on the same packed inputs:
fp32 outputs within max|diff| <= 1e-3 max|ref| and relative Frobenius <= 1e-4; bf16
outputs within one bf16 ulp of the rounded reference."""
import numpy as np
import pytest
import torch

from helpers import assert_bf16_rounding_of, assert_gemm_close
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def rand_e4m3(rng, shape):
    c = rng.integers(0, 0x7F, shape, dtype=np.uint8)          # no 0x7F (NaN)
    return c | (rng.integers(0, 2, shape, dtype=np.uint8) << 7)


def rand_mxfp8(rng, rows, k):
    return rand_e4m3(rng, (rows, k)), rng.integers(120, 135, (rows, k // 32), dtype=np.uint8)


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_mxfp8(F, a, asc, b, bsc, out_dtype=torch.float32):
    d = F.gemm_mxfp8(cu(a), cu(asc), cu(b), cu(bsc), out_dtype)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    return d


# ------------------------------------------------------------------ MXFP8
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (300, 272, 384), (1, 16, 128)])
def test_mxfp8_random_operands(F, orc, M, N, K):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    a, asc = rand_mxfp8(rng, M, K)
    b, bsc = rand_mxfp8(rng, N, K)
    d = run_mxfp8(F, a, asc, b, bsc)
    assert_gemm_close(d.cpu().numpy(), orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), f"MXFP8 {M}x{N}x{K}")


def test_mxfp8_structured_scales(F, orc):
    """All operands 1.0; scales vary by row, by column and by 32-block, so each lane,
    column and scale byte the tensor core reads is distinguishable."""
    M, N, K = 256, 512, 512
    a = np.full((M, K), 0x38, np.uint8)            # E4M3 1.0
    b = np.full((N, K), 0x38, np.uint8)
    asc = (127 + (np.arange(M)[:, None] % 5) + 0 * np.arange(K // 32)[None, :]).astype(np.uint8)
    bsc = (125 + (np.arange(K // 32)[None, :] % 4) + (np.arange(N)[:, None] % 3)).astype(np.uint8)
    d = run_mxfp8(F, a, asc, b, bsc)
    assert_gemm_close(d.cpu().numpy(), orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), "MXFP8 structured scales")


def test_mxfp8_bf16_output(F, orc):
    rng = np.random.default_rng(5)
    a, asc = rand_mxfp8(rng, 256, 512)
    b, bsc = rand_mxfp8(rng, 272, 512)
    d = run_mxfp8(F, a, asc, b, bsc, torch.bfloat16)
    got = d.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16_rounding_of(got, orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), "MXFP8 bf16 out")


def test_mxfp8_backward_from_requant(F, orc):
    """dgrad and wgrad of the backward-requant config, reduced to 512 tokens x 512 x 256,
    fed by the device requant (whose bytes equal the oracle's, tested elsewhere)."""
    M, K, N = 512, 512, 256
    seed, signs = I.sr_seed(2), I.rht_signs(2)
    dy = I.student_t(M, N, seed=2).cuda()
    x = I.normal_with_outliers(M, K, seed=22).cuda()
    w = I.normal(N, K, seed=23, std=0.02).cuda()
    xc, xs, xsd, _ = F.quantize_1d(x)
    wc, ws, wsd, _ = F.quantize_2d(w)
    wt = F.requant_mxfp8(F.IN_NVFP4_2D, wc, ws, wsd, N, K, 1, 0, 0, F.SR, seed, F.TAG_WT)
    g = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 0, 0, 0, F.SR, seed, F.TAG_DY_ROWS)
    gt = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 1, 1, signs, F.SR, seed, F.TAG_DY_T)
    xt = F.requant_mxfp8(F.IN_NVFP4_1D, xc, xs, xsd, M, K, 1, 1, signs, F.SR, seed, F.TAG_XT)
    dx = F.gemm_mxfp8(*g, *wt)
    dw = F.gemm_mxfp8(*gt, *xt)
    torch.cuda.synchronize()
    n = lambda t: t.cpu().numpy()
    assert_gemm_close(n(dx), orc.gemm_mxfp8(n(g[0]), n(g[1]), n(wt[0]), n(wt[1]), with_abs=True), "dgrad")
    assert_gemm_close(n(dw), orc.gemm_mxfp8(n(gt[0]), n(gt[1]), n(xt[0]), n(xt[1]), with_abs=True), "wgrad")
    # RHT cancels in the wgrad product: dW with rotated operands approximates dY^T X_q
    xq = orc.dequant_nvfp4(n(xc), n(xs), 1, float(xsd.item()))
    ref = dy.float().cpu().numpy().astype(np.float64).T @ xq
    rel = np.linalg.norm(n(dw) - ref) / np.linalg.norm(ref)
    assert rel < 0.1


# ------------------------------------------------------------------ NVFP4
def rand_nvfp4(rng, rows, k, two_d=False):
    codes = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    shape = (rows // 16, k // 16) if two_d else (rows, k // 16)
    return codes, rng.integers(0x18, 0x58, shape, dtype=np.uint8)


def run_nvfp4(F, a, asc, asd, b, bsc, bkind, bsd, out_dtype=torch.float32, groups=1, offs=None):
    d = F.gemm_nvfp4(cu(a), cu(asc), torch.tensor([asd], dtype=torch.float32, device="cuda"),
                     cu(b), cu(bsc), bkind, torch.tensor(np.atleast_1d(bsd), dtype=torch.float32, device="cuda"),
                     out_dtype, groups, offs)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    return d


@pytest.mark.parametrize("M,N,K,two_d", [(128, 256, 256, False), (256, 512, 1024, True),
                                          (300, 272, 768, False), (200, 48, 512, True), (1, 16, 256, True)])
def test_nvfp4_random_operands(F, orc, M, N, K, two_d):
    rng = np.random.default_rng(M + 3 * N + 5 * K)
    a, asc = rand_nvfp4(rng, M, K)
    b, bsc = rand_nvfp4(rng, N, K, two_d)
    asd, bsd = 0.375, float(np.float32(1 / 3))
    d = run_nvfp4(F, a, asc, asd, b, bsc, 2 if two_d else 1, bsd)
    ref = orc.gemm_nvfp4(a, asc, 1, asd, b, bsc, 2 if two_d else 1, bsd, with_abs=True)
    assert_gemm_close(d.cpu().numpy(), ref, f"NVFP4 {M}x{N}x{K} 2d={two_d}")


def test_nvfp4_structured_scales(F, orc):
    M, N, K = 256, 512, 1024
    a = np.full((M, K // 2), 0x22, np.uint8)                     # E2M1 1.0 in both nibbles
    b = np.full((N, K // 2), 0x22, np.uint8)
    kb = np.arange(K // 16)
    asc = (0x30 + (np.arange(M)[:, None] % 7) + 0 * kb[None, :]).astype(np.uint8)
    bsc = (0x2C + (kb[None, :] % 9) + (np.arange(N)[:, None] % 3)).astype(np.uint8)
    d = run_nvfp4(F, a, asc, 1.0, b, bsc, 1, 1.0)
    assert_gemm_close(d.cpu().numpy(), orc.gemm_nvfp4(a, asc, 1, 1.0, b, bsc, 1, 1.0, with_abs=True), "NVFP4 structured")


def test_nvfp4_bf16_output(F, orc):
    rng = np.random.default_rng(8)
    a, asc = rand_nvfp4(rng, 256, 512)
    b, bsc = rand_nvfp4(rng, 256, 512, True)
    d = run_nvfp4(F, a, asc, 0.5, b, bsc, 2, 0.25, torch.bfloat16)
    got = d.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16_rounding_of(got, orc.gemm_nvfp4(a, asc, 1, 0.5, b, bsc, 2, 0.25, with_abs=True), "NVFP4 bf16 out")


def test_nvfp4_grouped_equals_per_group(F, orc):
    rng = np.random.default_rng(9)
    G, N, K = 3, 272, 512
    rows = [100, 256, 37]
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    M = int(offs[-1])
    a, asc = rand_nvfp4(rng, M, K)
    bs = [rand_nvfp4(rng, N, K, True) for _ in range(G)]
    b = np.stack([x[0] for x in bs])
    bsc = np.stack([x[1] for x in bs])
    bsd = np.array([0.5, 0.25, 2.0], np.float32)
    d = run_nvfp4(F, a, asc, 1.0, b, bsc, 2, bsd, groups=G, offs=list(offs)).cpu().numpy()
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = orc.gemm_nvfp4(a[lo:hi], asc[lo:hi], 1, 1.0, b[g], bsc[g], 2, float(bsd[g]), with_abs=True)
        assert_gemm_close(d[lo:hi], ref, f"group {g}")


@pytest.mark.parametrize("two_d,out_dtype", [(True, torch.float32), (False, torch.float32), (True, torch.bfloat16)])
def test_nvfp4_grouped_pair_kernel(F, orc, two_d, out_dtype):
    """Grouped GEMMs on the persistent CTA-pair kernel (K a multiple of 1024): ragged groups, an
    empty group, groups smaller than a 128-row half tile, a ragged N."""
    rng = np.random.default_rng(17 + two_d)
    G, N, K = 5, 272, 1024
    rows = [300, 0, 37, 500, 256]
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    M = int(offs[-1])
    a, asc = rand_nvfp4(rng, M, K)
    bs = [rand_nvfp4(rng, N, K, two_d) for _ in range(G)]
    b = np.stack([x[0] for x in bs])
    bsc = np.stack([x[1] for x in bs])
    bsd = np.array([0.5, 0.25, 2.0, 1.0, 0.125], np.float32)
    d = run_nvfp4(F, a, asc, 0.75, b, bsc, 2 if two_d else 1, bsd, out_dtype, groups=G, offs=list(offs))
    got = d.float().cpu().numpy()
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        ref = orc.gemm_nvfp4(a[lo:hi], asc[lo:hi], 1, 0.75, b[g], bsc[g], 2 if two_d else 1, float(bsd[g]), with_abs=True)
        if out_dtype == torch.float32:
            assert_gemm_close(got[lo:hi], ref, f"pair group {g}")
        else:
            assert_bf16_rounding_of(d[lo:hi].cpu().view(torch.int16).numpy().view(np.uint16), ref, f"pair group {g}")


def test_nvfp4_single_linear_config(F, orc):
    """Config: X 256x512 (+outliers), W 256x512, Y = X W^T 256x256 fp32, seed 0."""
    x = I.normal_with_outliers(256, 512, seed=0)
    w = I.normal(256, 512, seed=100, std=0.02)
    xc, xs, xsd, _ = F.quantize_1d(x.cuda())
    wc, ws, wsd, _ = F.quantize_2d(w.cuda())
    y = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.float32)
    torch.cuda.synchronize()
    n = lambda t: t.cpu().numpy()
    ref = orc.gemm_nvfp4(n(xc), n(xs), 1, float(xsd.item()), n(wc), n(ws), 2, float(wsd.item()), with_abs=True)
    assert_gemm_close(n(y), ref, "single linear")
    # and the quantized layer approximates the bf16 layer (NVFP4 error ~10% per operand)
    full = x.float().numpy() @ w.float().numpy().T
    assert np.linalg.norm(n(y) - full) / np.linalg.norm(full) < 0.2


def test_nvfp4_moe_grouped_full_size(F, orc):
    """Config: 8 experts x 1024 tokens, K = 4096, N = 1536, bf16 out; sampled rows per expert."""
    E, T, K, N = 8, 8192, 4096, 1536
    x = I.normal_with_outliers(T, K, seed=1)
    w = torch.stack([I.normal(N, K, seed=1000 + e, std=0.02) for e in range(E)])
    xc, xs, xsd, _ = F.quantize_1d(x.cuda())
    wc, ws, wsd, _ = F.quantize_2d(w.cuda())
    offs = [e * (T // E) for e in range(E + 1)]
    y = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16, E, offs)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    yb = y.cpu().view(torch.int16).numpy().view(np.uint16)
    xc, xs, wc, ws = (t.cpu().numpy() for t in (xc, xs, wc, ws))
    for e in range(E):
        rows = np.arange(offs[e], offs[e + 1])[::128][:8] + (e * 13) % 100
        ref = orc.gemm_nvfp4(xc[rows], xs[rows], 1, float(xsd.item()), wc[e], ws[e], 2, float(wsd[e].item()), with_abs=True)
        assert_bf16_rounding_of(yb[rows], ref, f"expert {e}")


# ------------------------------------------------------------------ CTA-pair kernel (K >= 32 stages)
@pytest.mark.parametrize("M,N,K", [(300, 272, 4096), (512, 512, 4096), (129, 16, 4096)])
def test_mxfp8_pair_kernel_random(F, orc, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a, asc = rand_mxfp8(rng, M, K)
    b, bsc = rand_mxfp8(rng, N, K)
    d = run_mxfp8(F, a, asc, b, bsc)
    assert_gemm_close(d.cpu().numpy(), orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), f"MXFP8 pair {M}x{N}x{K}")


def test_mxfp8_pair_kernel_structured_scales(F, orc):
    M, N, K = 512, 512, 4096
    a = np.full((M, K), 0x38, np.uint8)
    b = np.full((N, K), 0x38, np.uint8)
    asc = (124 + (np.arange(M)[:, None] % 7) + (np.arange(K // 32)[None, :] % 2)).astype(np.uint8)
    bsc = (125 + (np.arange(K // 32)[None, :] % 4) + (np.arange(N)[:, None] // 32 % 3)).astype(np.uint8)
    d = run_mxfp8(F, a, asc, b, bsc, torch.bfloat16)
    got = d.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16_rounding_of(got, orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True), "MXFP8 pair structured, bf16 out")


# Many short tiles per cluster (512 tiles of 256 x 256 over 76 CTA pairs, 4 K-blocks each): the
# stage ring, the MXFP8 K-block groups and the tensor-memory scale slots wrap across tile
# boundaries, and each tile's epilogue overlaps the next tile's main loop. Every output compared.
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mxfp8_pair_kernel_many_short_tiles(F, orc, out_dtype):
    M, N, K = 8192, 4096, 512
    rng = np.random.default_rng(8192 + 512)
    a, asc = rand_mxfp8(rng, M, K)
    b, bsc = rand_mxfp8(rng, N, K)
    d = run_mxfp8(F, a, asc, b, bsc, out_dtype)
    ref = orc.gemm_mxfp8(a, asc, b, bsc, with_abs=True)
    if out_dtype == torch.float32:
        assert_gemm_close(d.cpu().numpy(), ref, f"MXFP8 pair {M}x{N}x{K}")
    else:
        assert_bf16_rounding_of(d.cpu().view(torch.int16).numpy().view(np.uint16), ref, f"MXFP8 pair {M}x{N}x{K} bf16")


@pytest.mark.parametrize("two_d", [False, True])
def test_nvfp4_pair_kernel_many_short_tiles(F, orc, two_d):
    M, N, K = 8192, 4096, 1024
    rng = np.random.default_rng(8192 + 1024 + two_d)
    a, asc = rand_nvfp4(rng, M, K)
    b, bsc = rand_nvfp4(rng, N, K, two_d)
    d = run_nvfp4(F, a, asc, 0.5, b, bsc, 2 if two_d else 1, 0.125)
    ref = orc.gemm_nvfp4(a, asc, 1, 0.5, b, bsc, 2 if two_d else 1, 0.125, with_abs=True)
    assert_gemm_close(d.cpu().numpy(), ref, f"NVFP4 pair {M}x{N}x{K} 2d={two_d}")


@pytest.mark.parametrize("M,N,K,two_d", [(300, 272, 8192, False), (256, 256, 8192, True)])
def test_nvfp4_pair_kernel_random(F, orc, M, N, K, two_d):
    rng = np.random.default_rng(M * 3 + N + K)
    a, asc = rand_nvfp4(rng, M, K)
    b, bsc = rand_nvfp4(rng, N, K, two_d)
    d = run_nvfp4(F, a, asc, 0.5, b, bsc, 2 if two_d else 1, 0.125)
    ref = orc.gemm_nvfp4(a, asc, 1, 0.5, b, bsc, 2 if two_d else 1, 0.125, with_abs=True)
    assert_gemm_close(d.cpu().numpy(), ref, f"NVFP4 pair {M}x{N}x{K} 2d={two_d}")
