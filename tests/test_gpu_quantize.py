"""NVFP4 quantize kernels (fp4q_quantize_1d / fp4q_quantize_2d) against the oracle:
packed codes, block scales, amax and s_dec bit for bit, on the configs' shapes and
distributions, ragged shapes, padded leading dimensions and degenerate tensors."""
import numpy as np
import pytest
import torch

from helpers import assert_bytes_equal
from mxfp8_precision_numerics_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def check_1d(F, orc, x, what, amax=None, ld_pad=0):
    rows, cols = x.shape
    if ld_pad:
        buf = torch.zeros(rows, cols + ld_pad, dtype=torch.bfloat16)
        buf[:, :cols] = x
        xd = buf.cuda()[:, :cols]
    else:
        xd = x.cuda()
    amax_in = None if amax is None else torch.tensor([amax], dtype=torch.float32, device="cuda")
    codes, scales, s_dec, amax_d = F.quantize_1d(xd, amax_in=amax_in)
    torch.cuda.synchronize()
    oc, os_, oa, osd = orc.quantize_1d(I.bf16_bits(x), amax=amax)
    assert_bytes_equal(codes.cpu().numpy(), oc, what + " codes")
    assert_bytes_equal(scales.cpu().numpy(), os_, what + " scales")
    assert float(s_dec.item()) == osd, what + " s_dec"
    assert float(amax_d.item()) == oa, what + " amax"
    return codes, scales, s_dec


def check_2d(F, orc, w, what):
    """w: [rows, cols] or [batch, rows, cols] bf16 (CPU)."""
    codes, tiles, s_dec, amax = F.quantize_2d(w.cuda())
    torch.cuda.synchronize()
    ws = w if w.dim() == 3 else w.unsqueeze(0)
    cs = codes if codes.dim() == 3 else codes.unsqueeze(0)
    ts = tiles if tiles.dim() == 3 else tiles.unsqueeze(0)
    for b in range(ws.shape[0]):
        oc, ot, oa, osd = orc.quantize_2d(I.bf16_bits(ws[b]))
        assert_bytes_equal(cs[b].cpu().numpy(), oc, f"{what}[{b}] codes")
        assert_bytes_equal(ts[b].cpu().numpy(), ot, f"{what}[{b}] tile scales")
        assert float(s_dec[b].item()) == osd, f"{what}[{b}] s_dec"
        assert float(amax[b].item()) == oa, f"{what}[{b}] amax"
    return codes, tiles, s_dec


# ------------------------------------------------------------------ 1D
def test_quantize_1d_single_linear_config(F, orc):
    check_1d(F, orc, I.normal_with_outliers(256, 512, seed=0), "X 256x512")


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (17, 272), (129, 4096 + 16)])
def test_quantize_1d_ragged_shapes(F, orc, rows, cols):
    check_1d(F, orc, I.normal_with_outliers(rows, cols, seed=rows * 7 + cols), f"X {rows}x{cols}")


def test_quantize_1d_padded_leading_dimension(F, orc):
    check_1d(F, orc, I.normal(40, 96, seed=3), "X 40x96 ld+24", ld_pad=24)


def test_quantize_1d_degenerate_tensors(F, orc):
    check_1d(F, orc, torch.zeros(16, 64, dtype=torch.bfloat16), "all-zero")
    # bf16 subnormals and a block far below the tensor max (scale clamps to 0x01)
    x = torch.zeros(8, 64, dtype=torch.float32)
    x[0, 0] = 3.0e4
    x[1, 16:32] = 1e-39
    x[2, 32:48] = -2.0e-3
    x[3, :] = torch.linspace(-1, 1, 64)
    check_1d(F, orc, x.to(torch.bfloat16), "subnormal / underflow")
    # every E2M1 tie: values exactly at midpoints once the block maps its max to 6
    ties = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -6.0, -0.25, -0.75, -1.25,
                         -1.75, -2.5, -3.5, -5.0], dtype=torch.float32)
    check_1d(F, orc, ties.repeat(4, 4).to(torch.bfloat16), "E2M1 ties", amax=2688.0)


def test_quantize_1d_given_amax_matches_sharded_run(F, orc):
    """Two row shards quantized with the agreed global amax equal the whole tensor."""
    x = I.normal_with_outliers(256, 512, seed=9)
    g_amax = float(x.float().abs().max())
    full_c, full_s, full_d = check_1d(F, orc, x, "whole")
    top_c, top_s, top_d = check_1d(F, orc, x[:128].contiguous(), "shard 0", amax=g_amax)
    bot_c, bot_s, bot_d = check_1d(F, orc, x[128:].contiguous(), "shard 1", amax=g_amax)
    assert torch.equal(torch.cat([top_c, bot_c]), full_c)
    assert torch.equal(torch.cat([top_s, bot_s]), full_s)
    assert float(top_d.item()) == float(full_d.item()) == float(bot_d.item())


def test_quantize_1d_moe_tokens_full_size(F, orc):
    check_1d(F, orc, I.normal_with_outliers(8192, 4096, seed=1), "X 8192x4096")


# ------------------------------------------------------------------ 2D
def test_quantize_2d_single_linear_config(F, orc):
    check_2d(F, orc, I.normal(256, 512, seed=100, std=0.02), "W 256x512")


@pytest.mark.parametrize("rows,cols", [(16, 16), (48, 272), (96, 4096 + 16)])
def test_quantize_2d_ragged_shapes(F, orc, rows, cols):
    check_2d(F, orc, I.normal_with_outliers(rows, cols, seed=rows + cols, std=0.02), f"W {rows}x{cols}")


def test_quantize_2d_transpose_invariance(F, orc):
    w = I.normal_with_outliers(64, 96, seed=5, std=0.02)
    c1, t1, d1 = check_2d(F, orc, w, "W")
    c2, t2, d2 = check_2d(F, orc, w.t().contiguous(), "W^T")
    assert torch.equal(t1.t(), t2)
    def unpack(c):
        c = c.cpu().numpy()
        out = np.empty((c.shape[0], c.shape[1] * 2), np.uint8)
        out[:, 0::2] = c & 15
        out[:, 1::2] = c >> 4
        return out
    assert np.array_equal(unpack(c1).T, unpack(c2))


def test_quantize_2d_moe_experts_full_size(F, orc):
    w = torch.stack([I.normal(1536, 4096, seed=1000 + e, std=0.02) for e in range(8)])
    check_2d(F, orc, w, "W_up 8x1536x4096")
