"""Full-size parity of the kernels the benchmark times, stage by stage.

* The GPT MLP block (tokens 16384, d_model 4096, ffn 16384; the benchmark's step, run by the
  same function, layer.mlp_step): every stage of one forward + backward is compared with the
  oracle on the GPU's own input for that stage, so an error shows where it starts. Packed
  codes and scales bit for bit on sampled rows; GEMM outputs on sampled rows x columns (each
  16-row group of a 16x16-scaled operand kept whole) against the oracle's float64 product of
  the same packed operands, by the criteria of tests/helpers.py; GELU / GELU' against the
  oracle's float64 functions of the GPU's own h; the epilogue's max|GELU(h)| exactly.
* The backward requantization workload (dY 8192 x 4096, X 8192 x 4096, W 4096 x 4096): the
  dgrad and the wgrad (4096 x 4096, K = 8192).
* The 2D weight quantize + GEMM sweep (W 14336 x 4096): the weight's codes and tile scales,
  and the GEMM at M = 1024, 4096 and 16384.

Seeded synthetic inputs as in the benchmark ("End-to-End 4-Bit Training" §13-14 for the MLP
block; "Pretraining Large Language Models with NVFP4", Quantization Procedure steps 1-5 and
the backward recipe)."""
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


def np_(t):
    return t.cpu().numpy()


def u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def sample_rows(n, k, seed):
    """k sorted distinct rows of n, always including the first and the last."""
    r = np.random.default_rng(seed).choice(n, k, replace=False)
    r[0], r[-1] = 0, n - 1
    return np.unique(r)


def sample_groups(n, g, seed):
    """g distinct whole 16-row groups of n rows (the first and the last among them), as
    (row indices, group indices)."""
    grp = np.random.default_rng(seed).choice(n // 16, g, replace=False)
    grp[0], grp[-1] = 0, n // 16 - 1
    grp = np.unique(grp)
    return (grp[:, None] * 16 + np.arange(16)[None, :]).reshape(-1), grp


def check_quantize_1d_rows(orc, x_bits, q, amax, rows, what):
    c, s, sd = q
    oc, os_, _, osd = orc.quantize_1d(x_bits[rows], amax=amax)
    assert float(sd.item()) == osd, what + " s_dec"
    idx = torch.from_numpy(rows).cuda()
    assert_bytes_equal(np_(c[idx]), oc, what + " codes")
    assert_bytes_equal(np_(s[idx]), os_, what + " scales")


def check_quantize_2d_groups(orc, w_bits, q, amax, grp_rows, grp, what):
    c, s, sd = q
    oc, os_, _, osd = orc.quantize_2d(w_bits[grp_rows], amax=amax)
    assert float(sd.reshape(-1)[0].item()) == osd, what + " s_dec"
    assert_bytes_equal(np_(c[torch.from_numpy(grp_rows).cuda()]), oc, what + " codes")
    assert_bytes_equal(np_(s[torch.from_numpy(grp).cuda()]), os_, what + " tile scales")


def check_requant(orc, got, kind, data, scales, s_dec, rows, cols, transpose, rht, signs, seed, tag, out_rows,
                  what):
    """Sampled output rows of a requantization, bit for bit (out_rows: a few (begin, end))."""
    e4, e8 = np_(got[0]), np_(got[1])
    for b, e in out_rows:
        r4, r8 = orc.requant_mxfp8(kind, data, scales, s_dec, rows, cols, transpose, rht, signs, orc.SR, seed,
                                   tag, out_rows=(b, e))
        assert_bytes_equal(e8[b:e], r8, f"{what} e8m0 rows {b}:{e}")
        assert_bytes_equal(e4[b:e], r4, f"{what} e4m3 rows {b}:{e}")


def out_ranges(n, seed):
    """Four ranges of 2 output rows: the first, the last and two inside."""
    r = np.random.default_rng(seed).integers(1, n // 2 - 1, 2) * 2
    return [(0, 2), (int(r[0]), int(r[0]) + 2), (int(r[1]), int(r[1]) + 2), (n - 2, n)]


# ------------------------------------------------------------------ the GPT MLP block
def test_gpt_mlp_block_stage_by_stage(F, orc):
    from mxfp8_precision_numerics_gb300 import layer
    M, D, Fh = 16384, 4096, 16384
    seed_cfg = 4
    x = I.normal_with_outliers(M, D, seed=seed_cfg)
    w1 = I.normal(Fh, D, seed=seed_cfg * 10 + 1, std=0.02)
    w2 = I.normal(D, Fh, seed=seed_cfg * 10 + 2, std=0.02)
    dy = I.student_t(M, D, seed=seed_cfg * 10 + 3)
    seed, signs = I.sr_seed(seed_cfg), I.rht_signs(seed_cfg)
    seed2 = seed ^ layer.SEED2_OFFSET
    xb, w1b, w2b, dyb = (I.bf16_bits(t) for t in (x, w1, w2, dy))
    S = layer.mlp_step(x.cuda(), w1.cuda(), w2.cuda(), dy.cuda(), seed, signs)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK

    R = sample_rows(M, 24, 1)                       # token rows of the GEMM outputs
    Rd = torch.from_numpy(R).cuda()
    # ---- forward quantizes (amax over the whole tensor, exact)
    x_amax = orc.amax_bf16(xb)
    assert float(S["x_amax"].item()) == x_amax
    check_quantize_1d_rows(orc, xb, S["xq"], x_amax, R, "X quantize_1d")
    w1_amax, w2_amax = orc.amax_bf16(w1b), orc.amax_bf16(w2b)
    assert float(S["w1_amax"].item()) == w1_amax and float(S["w2_amax"].item()) == w2_amax
    Cf, Cf_grp = sample_groups(Fh, 48, 2)           # ffn columns (W1 rows, whole 16-row groups)
    check_quantize_2d_groups(orc, w1b, S["w1q"], w1_amax, Cf, Cf_grp, "W1 quantize_2d")
    Cd, Cd_grp = sample_groups(D, 48, 3)            # d_model columns (W2 rows)
    check_quantize_2d_groups(orc, w2b, S["w2q"], w2_amax, Cd, Cd_grp, "W2 quantize_2d")

    # ---- layer 1: h = X_q W1_q^T with GELU in the epilogue (16384 x 16384, K = 4096)
    xc, xs, xsd = (np_(t) for t in S["xq"])
    w1c, w1s, w1d = S["w1q"]
    ref = orc.gemm_nvfp4(xc[R], xs[R], 1, float(xsd[0]), np_(w1c[torch.from_numpy(Cf).cuda()]),
                         np_(w1s[torch.from_numpy(Cf_grp).cuda()]), 2, float(w1d.item()), with_abs=True)
    h_s = u16(S["h"][Rd][:, torch.from_numpy(Cf).cuda()])
    assert_bf16_rounding_of(h_s, ref, "layer-1 h (GELU GEMM) sampled")
    a_s = u16(S["a"][Rd][:, torch.from_numpy(Cf).cuda()])
    assert_bf16_near(a_s, orc.gelu_bf16(h_s), 1, "GELU(h) sampled")
    # the epilogue's max|GELU(h)| over all 268M outputs: exactly the max of what it wrote
    a_max = float(S["a"].float().abs().max().item())
    assert float(S["a_amax"].item()) == a_max
    # every output of the first 256-row tile row (all 64 column tiles): GELU of the written h,
    # element for element
    tr = torch.arange(0, 256, device="cuda")
    full_h = u16(S["h"][tr])
    assert_bf16_near(u16(S["a"][tr]), orc.gelu_bf16(full_h), 1, "GELU(h) first tile row")

    # ---- layer 2's input: GELU(h) quantized with the epilogue's amax
    ab = u16(S["a"][Rd])
    ac, as_, ad = S["aq"]
    oc, os_, _, osd = orc.quantize_1d(ab, amax=a_max)
    assert float(ad.item()) == osd
    assert_bytes_equal(np_(ac[Rd]), oc, "GELU(h) quantize_1d codes")
    assert_bytes_equal(np_(as_[Rd]), os_, "GELU(h) quantize_1d scales")

    # ---- layer 2: y = A_q W2_q^T (16384 x 4096, K = 16384), bf16
    w2c, w2s, w2d = S["w2q"]
    ref = orc.gemm_nvfp4(oc, os_, 1, osd, np_(w2c[torch.from_numpy(Cd).cuda()]),
                         np_(w2s[torch.from_numpy(Cd_grp).cuda()]), 2, float(w2d.item()), with_abs=True)
    assert_bf16_rounding_of(u16(S["y"][Rd][:, torch.from_numpy(Cd).cuda()]), ref, "layer-2 y sampled")

    # ---- backward, layer 2: requantizations (bit for bit on sampled output rows)
    check_requant(orc, S["g"], orc.IN_BF16, dyb, None, 1.0, M, D, False, False, 0, seed, F.TAG_DY_ROWS,
                  out_ranges(M, 5), "dY rows")
    w2c_h, w2s_h = np_(w2c), np_(w2s)
    check_requant(orc, S["w2t"], orc.IN_NVFP4_2D, w2c_h, w2s_h, float(w2d.item()), D, Fh, True, False, 0, seed,
                  F.TAG_WT, out_ranges(Fh, 6), "W2_q^T")
    check_requant(orc, S["gt"], orc.IN_BF16, dyb, None, 1.0, M, D, True, True, signs, seed, F.TAG_DY_T,
                  out_ranges(D, 7), "dY^T rht")
    ac_h, as_h = np_(ac), np_(as_)
    check_requant(orc, S["at"], orc.IN_NVFP4_1D, ac_h, as_h, float(ad.item()), M, Fh, True, True, signs, seed,
                  F.TAG_XT, out_ranges(Fh, 8), "A_q^T rht")

    # ---- layer 2 dgrad with GELU' (16384 x 16384, K = 4096): the plain bf16 GEMM on the same
    # operands against the oracle, and dh = bf16(bf16(dA) GELU'(h)) against it
    g4, g8 = S["g"]
    t4, t8 = S["w2t"]
    da = F.gemm_mxfp8(g4, g8, t4, t8, torch.bfloat16)
    torch.cuda.synchronize()
    Cfd = torch.from_numpy(Cf).cuda()
    ref = orc.gemm_mxfp8(np_(g4[Rd]), np_(g8[Rd]), np_(t4[Cfd]), np_(t8[Cfd]), with_abs=True)
    da_s = u16(da[Rd][:, Cfd])
    assert_bf16_rounding_of(da_s, ref, "layer-2 dgrad sampled")
    want = bf16_values(da_s).astype(np.float64) * orc.gelu_bf16(h_s, grad=True)
    assert_bf16_near(u16(S["dh"][Rd][:, Cfd]), want, 2, "dh = dA GELU'(h) sampled")
    # whole first tile row of dh against the plain GEMM's bf16 output there
    want = bf16_values(u16(da[tr])).astype(np.float64) * orc.gelu_bf16(full_h, grad=True)
    assert_bf16_near(u16(S["dh"][tr]), want, 2, "dh first tile row")
    del da

    # ---- layer 2 wgrad: dW2 = dY^T_q A^T_q (4096 x 16384, K = 16384 tokens), fp32
    gt4, gt8 = S["gt"]
    at4, at8 = S["at"]
    Rw = sample_rows(D, 16, 9)
    Cw = sample_rows(Fh, 512, 10)
    ref = orc.gemm_mxfp8(np_(gt4[torch.from_numpy(Rw).cuda()]), np_(gt8[torch.from_numpy(Rw).cuda()]),
                         np_(at4[torch.from_numpy(Cw).cuda()]), np_(at8[torch.from_numpy(Cw).cuda()]), with_abs=True)
    assert_gemm_close(np_(S["dw2"][torch.from_numpy(Rw).cuda()][:, torch.from_numpy(Cw).cuda()]), ref,
                      "dW2 sampled")

    # ---- backward, layer 1: requantizations of dh (own seed) and of the saved operands
    dhb = u16(S["dh"])
    check_requant(orc, S["g1"], orc.IN_BF16, dhb, None, 1.0, M, Fh, False, False, 0, seed2, F.TAG_DY_ROWS,
                  out_ranges(M, 11), "dH rows")
    check_requant(orc, S["w1t"], orc.IN_NVFP4_2D, np_(w1c), np_(w1s), float(w1d.item()), Fh, D, True, False, 0,
                  seed2, F.TAG_WT, out_ranges(D, 12), "W1_q^T")
    check_requant(orc, S["g1t"], orc.IN_BF16, dhb, None, 1.0, M, Fh, True, True, signs, seed2, F.TAG_DY_T,
                  out_ranges(Fh, 13), "dH^T rht")
    check_requant(orc, S["xt"], orc.IN_NVFP4_1D, xc, xs, float(xsd[0]), M, D, True, True, signs, seed2,
                  F.TAG_XT, out_ranges(D, 14), "X_q^T rht")
    del dhb

    # ---- layer 1 dgrad: dX = dH_q W1^T_q (16384 x 4096, K = 16384), bf16
    g14, g18 = S["g1"]
    w14, w18 = S["w1t"]
    Cdd = torch.from_numpy(Cd).cuda()
    ref = orc.gemm_mxfp8(np_(g14[Rd]), np_(g18[Rd]), np_(w14[Cdd]), np_(w18[Cdd]), with_abs=True)
    assert_bf16_rounding_of(u16(S["dx"][Rd][:, Cdd]), ref, "dX sampled")

    # ---- layer 1 wgrad: dW1 = dH^T_q X^T_q (16384 x 4096, K = 16384 tokens), fp32
    h4, h8 = S["g1t"]
    x4, x8 = S["xt"]
    Rw = sample_rows(Fh, 16, 15)
    Cw = sample_rows(D, 512, 16)
    ref = orc.gemm_mxfp8(np_(h4[torch.from_numpy(Rw).cuda()]), np_(h8[torch.from_numpy(Rw).cuda()]),
                         np_(x4[torch.from_numpy(Cw).cuda()]), np_(x8[torch.from_numpy(Cw).cuda()]), with_abs=True)
    assert_gemm_close(np_(S["dw1"][torch.from_numpy(Rw).cuda()][:, torch.from_numpy(Cw).cuda()]), ref,
                      "dW1 sampled")


# ------------------------------------------------------------------ backward requantization config
def test_backward_requant_config_dgrad_and_wgrad(F, orc):
    """dY 8192 x 4096 Student-t(3) 1e-3, X 8192 x 4096 N(0,1), W 4096 x 4096 N(0,0.02):
    dgrad dX = dY_q W^T_q (8192 x 4096, K = 4096) and wgrad dW = dY^T_q X^T_q (4096 x 4096,
    K = 8192 tokens, fp32) on sampled rows x columns."""
    M, K, N = 8192, 4096, 4096
    seed, signs = I.sr_seed(2), I.rht_signs(2)
    dy = I.student_t(M, N, seed=2).cuda()
    x = I.normal(M, K, seed=22).cuda()
    w = I.normal(N, K, seed=23, std=0.02).cuda()
    xc, xs, xsd, _ = F.quantize_1d(x)
    wc, ws, wsd, _ = F.quantize_2d(w)
    g = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 0, 0, 0, F.SR, seed, F.TAG_DY_ROWS)
    wt = F.requant_mxfp8(F.IN_NVFP4_2D, wc, ws, wsd, N, K, 1, 0, 0, F.SR, seed, F.TAG_WT)
    gt = F.requant_mxfp8(F.IN_BF16, dy, None, None, M, N, 1, 1, signs, F.SR, seed, F.TAG_DY_T)
    xt = F.requant_mxfp8(F.IN_NVFP4_1D, xc, xs, xsd, M, K, 1, 1, signs, F.SR, seed, F.TAG_XT)
    dx32 = F.gemm_mxfp8(g[0], g[1], wt[0], wt[1], torch.float32)
    dx16 = F.gemm_mxfp8(g[0], g[1], wt[0], wt[1], torch.bfloat16)
    dw = F.gemm_mxfp8(gt[0], gt[1], xt[0], xt[1], torch.float32)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    # the bf16 output is the nearest-even bf16 of the fp32 output, bit for bit
    want16 = dx32.to(torch.bfloat16)
    assert torch.equal(dx16.view(torch.int16), want16.view(torch.int16))
    R = torch.from_numpy(sample_rows(M, 32, 21)).cuda()
    C = torch.from_numpy(sample_rows(K, 1024, 22)).cuda()
    ref = orc.gemm_mxfp8(np_(g[0][R]), np_(g[1][R]), np_(wt[0][C]), np_(wt[1][C]), with_abs=True)
    assert_gemm_close(np_(dx32[R][:, C]), ref, "dgrad 8192x4096x4096 sampled")
    assert_bf16_rounding_of(u16(dx16[R][:, C]), ref, "dgrad bf16 sampled")
    Rw = torch.from_numpy(sample_rows(N, 32, 23)).cuda()
    Cw = torch.from_numpy(sample_rows(K, 1024, 24)).cuda()
    ref = orc.gemm_mxfp8(np_(gt[0][Rw]), np_(gt[1][Rw]), np_(xt[0][Cw]), np_(xt[1][Cw]), with_abs=True)
    assert_gemm_close(np_(dw[Rw][:, Cw]), ref, "wgrad 4096x4096x8192 sampled")


# ------------------------------------------------------------------ 2D weight quantize + GEMM sweep
@pytest.fixture(scope="module")
def sweep_weight(F):
    w = I.normal(14336, 4096, seed=33, std=0.02)
    wc, ws, wsd, wa = F.quantize_2d(w.cuda())
    torch.cuda.synchronize()
    return I.bf16_bits(w), (wc, ws, wsd), wa


def test_sweep_weight_quantize_2d_full_size(F, orc, sweep_weight):
    wb, wq, wa = sweep_weight
    amax = orc.amax_bf16(wb)
    assert float(wa.item()) == amax
    rows, grp = sample_groups(14336, 64, 31)
    check_quantize_2d_groups(orc, wb, wq, amax, rows, grp, "W 14336x4096 quantize_2d")


@pytest.mark.parametrize("M", [1024, 4096, 16384])
def test_sweep_gemm_sampled(F, orc, sweep_weight, M):
    """X M x 4096 N(0,1), W 14336 x 4096 (16x16 tiles), bf16 out; the fp32 output of the same
    GEMM checked too, and the bf16 output equal to its nearest-even rounding."""
    K, N = 4096, 14336
    _, (wc, ws, wsd), _ = sweep_weight
    x = I.normal(M, K, seed=3)
    xc, xs, xsd, _ = F.quantize_1d(x.cuda())
    y16 = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.bfloat16)
    y32 = F.gemm_nvfp4(xc, xs, xsd, wc, ws, F.SCALE_2D, wsd, torch.float32)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
    R = torch.from_numpy(sample_rows(M, 32, 40 + M)).cuda()
    Cr, Cg = sample_groups(N, 64, 41)
    C = torch.from_numpy(Cr).cuda()
    ref = orc.gemm_nvfp4(np_(xc[R]), np_(xs[R]), 1, float(xsd.item()), np_(wc[C]),
                         np_(ws[torch.from_numpy(Cg).cuda()]), 2, float(wsd.item()), with_abs=True)
    assert_gemm_close(np_(y32[R][:, C]), ref, f"C4 M={M} fp32 sampled")
    assert_bf16_rounding_of(u16(y16[R][:, C]), ref, f"C4 M={M} bf16 sampled")
