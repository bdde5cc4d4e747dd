"""The MoE combine wire format (4bit.vizuara.ai §11: RHT32 + block-scaled S2F6) against the
oracle, bit for bit: fp4q_combine_encode on fp32 and bf16 inputs (ragged, heavy-tailed,
degenerate and full-size sampled rows), fp4q_combine_decode with several arrivals per token,
and the NVFP4 GEMM whose epilogue writes the wire format (grouped and CTA-pair kernels), which
must equal the stand-alone encoder applied to the same GEMM's fp32 output."""
import numpy as np
import pytest
import torch

from helpers import assert_bytes_equal
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SIGNS = 0x9E37_79B9


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_encode(F, orc, x, what, signs=SIGNS):
    """x: CPU fp32 or bf16 tensor."""
    codes, e8 = F.combine_encode(x.cuda(), signs)
    torch.cuda.synchronize()
    if x.dtype == torch.bfloat16:
        oc, oe = orc.combine_encode(I.bf16_bits(x), signs, is_bf16=True)
    else:
        oc, oe = orc.combine_encode(x.numpy(), signs)
    assert_bytes_equal(e8.cpu().numpy(), oe, what + " e8m0")
    assert_bytes_equal(codes.cpu().numpy(), oc, what + " codes")
    return codes, e8


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 96), (65, 4096 + 32), (300, 256)])
def test_encode_shapes(F, orc, rows, cols, dtype):
    x = I.student_t(rows, cols, seed=rows + cols, df=3, scale=1.0).float().to(dtype)
    check_encode(F, orc, x, f"encode {rows}x{cols} {dtype}")


def test_encode_degenerate_values(F, orc):
    x = torch.zeros(8, 64, dtype=torch.float32)
    x[1, :] = 1e30
    x[1, 5] = -3e38                      # exponent clamped at 127: codes saturate
    x[2, :32] = 1e-39                    # subnormal inputs
    x[3, 7] = 1e-41
    x[4, :] = torch.linspace(-2.0, 127 / 64, 64)
    x[5, ::3] = -1.0
    x[6, :] = 1.0 / 64
    x[7, 0] = 5.0
    for signs in (0, SIGNS, 0xFFFF_FFFF):
        check_encode(F, orc, x, f"degenerate signs={signs:#x}", signs)


def check_decode(F, orc, tokens, k, cols, out_dtype, seed, e8m0_offset=0):
    x = I.student_t(tokens * k, cols, seed=seed, df=3, scale=1.0).float()
    oc, oe = orc.combine_encode(x.numpy(), SIGNS)
    e8 = cu(oe)
    if e8m0_offset:                      # the same scales at an address that is not 4-byte aligned
        buf = torch.zeros(oe.size + e8m0_offset, dtype=torch.uint8, device="cuda")
        buf[e8m0_offset:] = e8.flatten()
        e8 = buf[e8m0_offset:].view(oe.shape)
        assert e8.data_ptr() % 4 != 0
    out = F.combine_decode(cu(oc), e8, k, SIGNS, out_dtype)
    torch.cuda.synchronize()
    ref = orc.combine_decode(oc, oe, k, SIGNS)
    if out_dtype == torch.bfloat16:
        ref = orc.round_bf16(ref)
    got = out.float().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32)), \
        f"decode differs: tokens {tokens} k {k} cols {cols} {out_dtype}"


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols", [160, 1024])
def test_decode_sums_arrivals(F, orc, k, out_dtype, cols):
    """cols 160: one thread per group; cols 1024: the staged kernel (32-group chunks)."""
    check_decode(F, orc, 37, k, cols, out_dtype, seed=10 + k)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_many_arrivals_and_unaligned_scales(F, orc, out_dtype):
    """k = 8 (staged for bf16 output; fp32 output's ring would not fit, so the per-thread
    kernel), k = 7 (staged for both), and scales at an odd address (per-thread kernel)."""
    check_decode(F, orc, 9, 8, 2048, out_dtype, seed=31)
    check_decode(F, orc, 11, 7, 1024, out_dtype, seed=32)
    check_decode(F, orc, 13, 2, 1024, out_dtype, seed=33, e8m0_offset=1)


def test_combine_full_size_sampled(F, orc):
    """MoE combine at the MoE layer's size: 8192 tokens x d_model 4096, two arrivals each."""
    tokens, k, cols = 8192, 2, 4096
    x = I.student_t(tokens * k, cols, seed=21, df=3, scale=1.0).float()
    codes, e8 = F.combine_encode(x.cuda(), SIGNS)
    out = F.combine_decode(codes, e8, k, SIGNS, torch.float32)
    torch.cuda.synchronize()
    pick = np.array([0, 1, 4095, 8191])
    rows = np.concatenate([[t * k + j for j in range(k)] for t in pick])
    oc, oe = orc.combine_encode(x.numpy()[rows], SIGNS)
    assert_bytes_equal(codes.cpu().numpy()[rows], oc, "codes")
    assert_bytes_equal(e8.cpu().numpy()[rows], oe, "e8m0")
    ref = orc.combine_decode(oc, oe, k, SIGNS)
    assert np.array_equal(out.cpu().numpy()[pick], ref)


# ------------------------------------------------------------------ the GEMM with the encode epilogue
def rand_nvfp4(rng, rows, k, two_d=False):
    codes = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    shape = (rows // 16, k // 16) if two_d else (rows, k // 16)
    return codes, rng.integers(0x18, 0x58, shape, dtype=np.uint8)


@pytest.mark.parametrize("M,N,K,groups", [(300, 256, 512, 1), (512, 512, 4096, 1), (260, 96, 512, 3),
                                          (100, 64, 256, 1), (260, 288, 1024, 3)])
def test_gemm_combine_epilogue(F, orc, M, N, K, groups):
    """The fused encode equals fp4q_combine_encode of the plain GEMM's fp32 output (same
    accumulators), and the oracle's encode of that output. Single-CTA kernel (K < 1024 or
    M <= 128), CTA-pair kernel (K a multiple of 1024), grouped on both."""
    rng = np.random.default_rng(M + N + K)
    a, asc = rand_nvfp4(rng, M, K)
    asd = torch.tensor([0.375], dtype=torch.float32, device="cuda")
    if groups == 1:
        b, bsc = rand_nvfp4(rng, N, K, True)
        offs = None
        bsd = torch.tensor([float(np.float32(1 / 3))], dtype=torch.float32, device="cuda")
    else:
        bs = [rand_nvfp4(rng, N, K, True) for _ in range(groups)]
        b, bsc = np.stack([c for c, _ in bs]), np.stack([s for _, s in bs])
        offs = [0, 100, 100, M]
        bsd = torch.tensor([0.5, 0.25, 2.0], dtype=torch.float32, device="cuda")
    d = F.gemm_nvfp4(cu(a), cu(asc), asd, cu(b), cu(bsc), F.SCALE_2D, bsd, torch.float32, groups, offs)
    codes, e8 = F.gemm_nvfp4_combine(cu(a), cu(asc), asd, cu(b), cu(bsc), F.SCALE_2D, bsd, SIGNS, groups, offs)
    rc, re = F.combine_encode(d, SIGNS)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert_bytes_equal(e8.cpu().numpy(), re.cpu().numpy(), "fused e8m0 vs encode(GEMM)")
    assert_bytes_equal(codes.cpu().numpy(), rc.cpu().numpy(), "fused codes vs encode(GEMM)")
    oc, oe = orc.combine_encode(d.cpu().numpy(), SIGNS)
    assert_bytes_equal(codes.cpu().numpy(), oc, "fused codes vs oracle")
    assert_bytes_equal(e8.cpu().numpy(), oe, "fused e8m0 vs oracle")
