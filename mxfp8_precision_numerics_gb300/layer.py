"""The NVFP4 linear layer and GPT MLP block, composed from the fp4q entry points.

Forward (4bit.vizuara.ai §10 figure; "Pretraining Large Language Models with NVFP4"):
activations are quantized to NVFP4 with 1x16 blocks, weights with 16x16 tiles, and one
NVFP4 GEMM produces the output. Only the quantized tensors are saved.

Backward: the output gradient is quantized to MXFP8 with stochastic rounding twice —
as it is for dgrad and transposed (with the 16-point RHT) for wgrad; the saved NVFP4
weight and activation are dequantized, transposed and re-quantized to MXFP8 with SR
(the activation with the RHT, the weight without). dgrad sums over N, wgrad over tokens.

Activations take either one outer scale per tensor (the NVFP4 paper's recipe) or, with
outer="row", one per token row plus the Four Over Six block-scale choice (4bit.vizuara.ai §10:
QLinearFn quantizes x with outer="row", four_six=True and w with outer="tensor").

GELU between the two linear layers of the MLP block (exact erf form, bf16) is fused into the
epilogues of the GEMMs around it: the first layer's NVFP4 GEMM writes h, GELU(h) and
max|GELU(h)| (which the second layer's quantize takes as its amax), and the second layer's
dgrad GEMM multiplies by GELU'(h) before writing dL/dh. Every quantize, requantize, transform,
GEMM and activation runs in libfp4q.
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
    x_rows: bool = False   # xq's s_dec holds one outer scale per row


def linear_forward(x, w=None, wq=None, out_dtype=torch.bfloat16, stream=None, x_amax=None, gelu=False,
                   outer="tensor", four_six=True):
    """y = x w^T on NVFP4 operands. x: [M, K] bf16; w: [N, K] bf16 (or wq precomputed).
    outer: "tensor" (one outer scale for x; x_amax = max|x| if already known, as a device
    float) or "row" (one per token row, with 4/6 block scales if four_six).
    gelu=True returns ((h, GELU(h), max|GELU(h)|), saved) instead of (y, saved); with
    outer="row" it returns ((h, GELU(h)), saved)."""
    if outer not in ("tensor", "row"):
        raise ValueError(f"outer must be 'tensor' or 'row', not {outer!r}")
    rows = outer == "row"
    M, K = x.shape
    if rows:
        xc, xs, xsd = F.quantize_1d_rows(x, four_six, stream=stream)
    else:
        xc, xs, xsd, _ = F.quantize_1d(x, amax_in=x_amax, stream=stream)
    if wq is None:
        wc, ws, wsd, _ = F.quantize_2d(w, stream=stream)
        wq = (wc, ws, wsd)
    wc, ws, wsd = wq
    N = wc.shape[0]
    saved = SavedLinear((xc, xs, xsd), wq, M, K, N, rows)
    if gelu:
        fn = F.gemm_nvfp4_gelu_rows if rows else F.gemm_nvfp4_gelu
        return fn(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, stream=stream), saved
    fn = F.gemm_nvfp4_rows if rows else F.gemm_nvfp4
    y = fn(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, out_dtype, stream=stream)
    return y, saved


def linear_backward(dy, saved, seed, rht_signs, dx_dtype=torch.bfloat16, stream=None,
                    rounding=F.SR, dgelu_h=None):
    """dy: [M, N] bf16 -> (dx [M, K], dw [N, K] fp32). dgelu_h: the previous layer's
    pre-activation h; when given, dx is returned as dx * GELU'(h) (bf16)."""
    M, K, N = saved.M, saved.K, saved.N
    xc, xs, xsd = saved.xq
    wc, ws, wsd = saved.wq
    # dy's two quantizations from one read: rowwise (blocks along N) for dgrad, transposed with
    # the RHT (blocks and transform along tokens) for wgrad
    g, gt = F.requant_bf16_dual(dy, 1, rht_signs, rounding, seed, F.TAG_DY_ROWS, F.TAG_DY_T, stream)
    # dgrad: dx[m, k] = sum_n dy[m, n] w[n, k]   (blocks along N on both operands)
    wt = F.requant_mxfp8(F.IN_NVFP4_2D, wc, ws, wsd, N, K, 1, 0, 0, rounding, seed, F.TAG_WT, stream)
    if dgelu_h is not None:
        dx = F.gemm_mxfp8_dgelu(g[0], g[1], wt[0], wt[1], dgelu_h, stream)
    else:
        dx = F.gemm_mxfp8(g[0], g[1], wt[0], wt[1], dx_dtype, stream)
    # wgrad: dw[n, k] = sum_m dy[m, n] x[m, k]   (blocks and RHT along tokens)
    x_kind = F.IN_NVFP4_1D_ROWS if saved.x_rows else F.IN_NVFP4_1D
    xt = F.requant_mxfp8(x_kind, xc, xs, xsd, M, K, 1, 1, rht_signs, rounding, seed, F.TAG_XT, stream)
    dw = F.gemm_mxfp8(gt[0], gt[1], xt[0], xt[1], torch.float32, stream)
    return dx, dw


def mlp_forward(x, w1, w2, stream=None, outer="tensor"):
    """GPT MLP block: y = gelu(x w1^T) w2^T. x [M, D], w1 [Fh, D], w2 [D, Fh].
    outer="row": both activations (x and GELU(h)) per token row with 4/6 block scales."""
    if outer == "row":
        (h, a), s1 = linear_forward(x, w1, stream=stream, gelu=True, outer="row")
        y, s2 = linear_forward(a, w2, stream=stream, outer="row")
        return y, (h, s1, s2)
    (h, a, a_amax), s1 = linear_forward(x, w1, stream=stream, gelu=True)
    y, s2 = linear_forward(a, w2, stream=stream, x_amax=a_amax)
    return y, (h, s1, s2)


def mlp_backward(dy, saved, seed, rht_signs, stream=None):
    h, s1, s2 = saved
    # layer 2's dgrad GEMM applies GELU'(h): dh = (dy w2) * GELU'(h)
    dh, dw2 = linear_backward(dy, s2, seed, rht_signs, stream=stream, dgelu_h=h)
    # a second layer draws from its own counter stream: offset the seed
    dx, dw1 = linear_backward(dh, s1, seed ^ SEED2_OFFSET, rht_signs, stream=stream)
    return dx, dw1, dw2


SEED2_OFFSET = 0x9E3779B97F4A7C15   # the second layer's counter stream: seed ^ this


def _direct(kind, units, fn, *a, **k):
    return fn(*a, **k)


def mlp_step(x, w1, w2, dy, seed, rht_signs, outer="tensor", call=None):
    """One forward + backward of the GPT MLP block, call by call, returning every stage's
    output in a dict (the same calls as mlp_forward + mlp_backward, with the intermediates
    kept so that each can be checked on its own input).

    x [M, D], w1 [Fh, D], w2 [D, Fh], dy [M, D], all bf16. outer: "tensor" or "row" (the
    activations x and GELU(h) per token row with 4/6 block scales). call(kind, units, fn,
    *args, **kwargs) runs each library call (default: directly); kind names the call's class
    and units its algorithmic size: elements for the HBM-bound calls, FLOPs for the GEMMs.
    """
    C = call or _direct
    M, D = x.shape
    Fh = w1.shape[0]
    rows = outer == "row"
    x_kind = F.IN_NVFP4_1D_ROWS if rows else F.IN_NVFP4_1D
    S = {}
    # ---- forward
    if rows:
        S["xq"] = C("quantize_1d_rows46", M * D, F.quantize_1d_rows, x, True)
    else:
        xc, xs, xsd, xa = C("quantize_1d", M * D, F.quantize_1d, x)
        S["xq"], S["x_amax"] = (xc, xs, xsd), xa
    w1c, w1s, w1d, w1a = C("quantize_2d", Fh * D, F.quantize_2d, w1)
    S["w1q"], S["w1_amax"] = (w1c, w1s, w1d), w1a
    xc, xs, xsd = S["xq"]
    # layer 1 with GELU in its epilogue: h, a = GELU(h) (and max|a|, layer 2's quantize amax)
    if rows:
        S["h"], S["a"] = C("gemm_nvfp4", 2.0 * M * Fh * D, F.gemm_nvfp4_gelu_rows, xc, xs, xsd, w1c, w1s,
                           F.SCALE_2D, w1d)
        S["aq"] = C("quantize_1d_rows46", M * Fh, F.quantize_1d_rows, S["a"], True)
    else:
        S["h"], S["a"], S["a_amax"] = C("gemm_nvfp4", 2.0 * M * Fh * D, F.gemm_nvfp4_gelu, xc, xs, xsd, w1c, w1s,
                                        F.SCALE_2D, w1d)
        ac, as_, ad, _ = C("quantize_1d_given_amax", M * Fh, F.quantize_1d, S["a"], amax_in=S["a_amax"])
        S["aq"] = (ac, as_, ad)
    w2c, w2s, w2d, w2a = C("quantize_2d", D * Fh, F.quantize_2d, w2)
    S["w2q"], S["w2_amax"] = (w2c, w2s, w2d), w2a
    ac, as_, ad = S["aq"]
    gemm2 = F.gemm_nvfp4_rows if rows else F.gemm_nvfp4
    S["y"] = C("gemm_nvfp4", 2.0 * M * D * Fh, gemm2, ac, as_, ad, w2c, w2s, F.SCALE_2D, w2d, torch.bfloat16)
    # ---- backward, layer 2: dA = dY W2 (times GELU'(h) in the epilogue), dW2 = dY^T A_q
    sr = F.SR
    # dY's two quantizations (rowwise for dgrad; transposed with the RHT for wgrad) from one read
    S["g"], S["gt"] = C("requant_bf16_dual", M * D, F.requant_bf16_dual, dy, 1, rht_signs, sr, seed,
                        F.TAG_DY_ROWS, F.TAG_DY_T)
    S["w2t"] = C("requant_nvfp4_2d", D * Fh, F.requant_mxfp8, F.IN_NVFP4_2D, w2c, w2s, w2d, D, Fh, 1, 0, 0, sr,
                 seed, F.TAG_WT)
    S["dh"] = C("gemm_mxfp8", 2.0 * M * Fh * D, F.gemm_mxfp8_dgelu, *S["g"], *S["w2t"], S["h"])
    S["at"] = C("requant_nvfp4_1d", M * Fh, F.requant_mxfp8, x_kind, ac, as_, ad, M, Fh, 1, 1, rht_signs, sr,
                seed, F.TAG_XT)
    S["dw2"] = C("gemm_mxfp8", 2.0 * D * Fh * M, F.gemm_mxfp8, *S["gt"], *S["at"], torch.float32)
    # ---- backward, layer 1: dX = dH W1, dW1 = dH^T X_q (its own counter stream)
    seed2 = seed ^ SEED2_OFFSET
    S["g1"], S["g1t"] = C("requant_bf16_dual", M * Fh, F.requant_bf16_dual, S["dh"], 1, rht_signs, sr, seed2,
                          F.TAG_DY_ROWS, F.TAG_DY_T)
    S["w1t"] = C("requant_nvfp4_2d", Fh * D, F.requant_mxfp8, F.IN_NVFP4_2D, w1c, w1s, w1d, Fh, D, 1, 0, 0, sr,
                 seed2, F.TAG_WT)
    S["dx"] = C("gemm_mxfp8", 2.0 * M * D * Fh, F.gemm_mxfp8, *S["g1"], *S["w1t"], torch.bfloat16)
    S["xt"] = C("requant_nvfp4_1d", M * D, F.requant_mxfp8, x_kind, xc, xs, xsd, M, D, 1, 1, rht_signs, sr,
                seed2, F.TAG_XT)
    S["dw1"] = C("gemm_mxfp8", 2.0 * Fh * D * M, F.gemm_mxfp8, *S["g1t"], *S["xt"], torch.float32)
    return S


def mlp_gemm_flops(M, D, Fh):
    """Dense GEMM FLOPs of one forward + backward pass: 2 NVFP4 + 4 MXFP8 GEMMs."""
    return 6 * 2 * M * D * Fh


def mlp_kernel_launches(outer="tensor"):
    """libfp4q kernels one mlp_forward + mlp_backward launches (counted from the calls):
    forward: amax + quantize_1d of x, quantize_1d of GELU(h) (its amax comes from the GELU
    GEMM's epilogue), 2 x (amax + quantize_2d of a weight), 2 NVFP4 GEMMs = 9 (outer="row":
    one per-row quantize for each activation, no activation amax: 8);
    backward: 2 x (3 requant, one of them the output gradient's two quantizations from one read,
    + 2 MXFP8 GEMMs) = 10."""
    return 18 if outer == "row" else 19
