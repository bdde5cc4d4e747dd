"""The NVFP4 linear layer and GPT MLP block, composed from the fp4q entry points.

Forward (4bit.vizuara.ai §10 figure; "Pretraining Large Language Models with NVFP4"):
activations are quantized to NVFP4 with 1x16 blocks, weights with 16x16 tiles, and one
NVFP4 GEMM produces the output. Only the quantized tensors are saved.

Backward: the output gradient is quantized to MXFP8 with stochastic rounding twice —
as it is for dgrad and transposed (with the 16-point RHT) for wgrad; the saved NVFP4
weight and activation are dequantized, transposed and re-quantized to MXFP8 with SR
(the activation with the RHT, the weight without). dgrad sums over N, wgrad over tokens.

GELU and its derivative between the two linear layers of the MLP block run in PyTorch
(bf16, exact erf form): they are the block's glue, not part of the quantized path.
Every quantize, requantize, transform and GEMM runs in libfp4q.
"""
from dataclasses import dataclass

import torch

from . import fp4q as F


@dataclass
class SavedLinear:
    xq: tuple          # (codes, scales, s_dec) of the input, 1D blocks
    wq: tuple          # (codes, tile scales, s_dec) of the weight, 16x16 tiles
    M: int
    K: int
    N: int


def linear_forward(x, w=None, wq=None, out_dtype=torch.bfloat16, stream=None):
    """y = x w^T on NVFP4 operands. x: [M, K] bf16; w: [N, K] bf16 (or wq precomputed)."""
    M, K = x.shape
    xc, xs, xsd, _ = F.quantize_1d(x, stream=stream)
    if wq is None:
        wc, ws, wsd, _ = F.quantize_2d(w, stream=stream)
        wq = (wc, ws, wsd)
    wc, ws, wsd = wq
    N = wc.shape[0]
    y = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, out_dtype, stream=stream)
    return y, SavedLinear((xc, xs, xsd), wq, M, K, N)


def linear_backward(dy, saved, seed, rht_signs, dx_dtype=torch.bfloat16, stream=None,
                    rounding=F.SR):
    """dy: [M, N] bf16 -> (dx [M, K], dw [N, K] fp32)."""
    M, K, N = saved.M, saved.K, saved.N
    xc, xs, xsd = saved.xq
    wc, ws, wsd = saved.wq
    # dgrad: dx[m, k] = sum_n dy[m, n] w[n, k]   (blocks along N on both operands)
    g = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 0, 0, 0, rounding, seed, F.TAG_DY_ROWS, stream)
    wt = F.requant_mxfp8(F.IN_NVFP4_2D, wc, ws, wsd, N, K, 1, 0, 0, rounding, seed, F.TAG_WT, stream)
    dx = F.gemm_mxfp8(g[0], g[1], wt[0], wt[1], dx_dtype, stream)
    # wgrad: dw[n, k] = sum_m dy[m, n] x[m, k]   (blocks and RHT along tokens)
    gt = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 1, 1, rht_signs, rounding, seed, F.TAG_DY_T, stream)
    xt = F.requant_mxfp8(F.IN_NVFP4_1D, xc, xs, xsd, M, K, 1, 1, rht_signs, rounding, seed, F.TAG_XT, stream)
    dw = F.gemm_mxfp8(gt[0], gt[1], xt[0], xt[1], torch.float32, stream)
    return dx, dw


def mlp_forward(x, w1, w2, stream=None):
    """GPT MLP block: y = gelu(x w1^T) w2^T. x [M, D], w1 [Fh, D], w2 [D, Fh]."""
    h, s1 = linear_forward(x, w1, stream=stream)
    a = torch.nn.functional.gelu(h)
    y, s2 = linear_forward(a, w2, stream=stream)
    return y, (h, s1, s2)


def mlp_backward(dy, saved, seed, rht_signs, stream=None):
    h, s1, s2 = saved
    da, dw2 = linear_backward(dy, s2, seed, rht_signs, stream=stream)
    dh = torch.ops.aten.gelu_backward(da, h)
    # a second layer draws from its own counter stream: offset the seed
    dx, dw1 = linear_backward(dh, s1, seed ^ 0x9E3779B97F4A7C15, rht_signs, stream=stream)
    return dx, dw1, dw2


def mlp_gemm_flops(M, D, Fh):
    """Dense GEMM FLOPs of one forward + backward pass: 2 NVFP4 + 4 MXFP8 GEMMs."""
    return 6 * 2 * M * D * Fh


def mlp_kernel_launches():
    """libfp4q kernels one mlp_forward + mlp_backward launches (counted from the calls):
    forward: 2 x (amax + quantize_1d, amax + quantize_2d, NVFP4 GEMM) = 10;
    backward: 2 x (4 requant + 2 MXFP8 GEMM) = 12."""
    return 22
