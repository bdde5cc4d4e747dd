"""Pins for the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a value the
pages print (fixtures under tests/golden/, each with its citation), a closed form,
an invariant, a special case with an exact answer, or a statistical law.
"""
import math

import numpy as np
import pytest

from conftest import read_golden_rows
from mxfp8_precision_numerics_gb300 import inputs

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16(values):
    """float list -> bf16 bit patterns (round to nearest even), shape kept."""
    import torch
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return inputs.bf16_bits(t)


def unpack_codes(codes):
    lo = codes & 0x0F
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


# ------------------------------------------------------------------ E2M1
def test_e2m1_decode_matches_page_table(orc):
    rows = read_golden_rows("e2m1_table.txt")
    assert len(rows) == 16
    for code, value in rows:
        v = orc.e2m1_decode(int(code))
        assert v == float(value)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(value))
    assert orc.e2m1_decode(0b0111) == 6.0


def test_e2m1_encode_page_examples(orc, worked):
    assert orc.e2m1_decode(orc.e2m1_encode_rne(worked["rtn_3p2"]["x"])) == worked["rtn_3p2"]["q"]
    ex = worked["rtn_5p4"]
    t = np.float32(ex["x"]) / np.float32(ex["scale"])
    assert orc.e2m1_decode(orc.e2m1_encode_rne(t)) == ex["q"]
    assert orc.e2m1_decode(orc.e2m1_encode_rne(t)) * ex["scale"] == ex["deq"]
    # 2.25 to nearest is 2 (the deterministic choice the SR example contrasts with)
    assert orc.e2m1_decode(orc.e2m1_encode_rne(2.25)) == 2.0


def test_e2m1_ties_go_to_even_code_and_sign_is_kept(orc):
    for i in range(7):
        mid = (E2M1_GRID[i] + E2M1_GRID[i + 1]) / 2
        lo_code, hi_code = i, i + 1
        want = lo_code if lo_code % 2 == 0 else hi_code
        assert orc.e2m1_encode_rne(mid) == want, mid
        assert orc.e2m1_encode_rne(-mid) == 8 | want, -mid
        # just off the midpoint the nearest value wins
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(100))
        assert orc.e2m1_encode_rne(below) == lo_code
        assert orc.e2m1_encode_rne(above) == hi_code
    assert orc.e2m1_encode_rne(-0.1) == 0x8          # rounds to zero, keeps the sign
    assert orc.e2m1_encode_rne(-0.0) == 0x8
    assert orc.e2m1_encode_rne(1e30) == 0x7          # saturates at 6
    assert orc.e2m1_encode_rne(-7.0) == 0xF


def test_e2m1_encode_is_monotone_and_within_half_gap(orc):
    xs = np.linspace(-7.0, 7.0, 20001, dtype=np.float32)
    prev = -1e9
    for x in xs:
        q = orc.e2m1_decode(orc.e2m1_encode_rne(x))
        assert q >= prev
        prev = q
        a = min(abs(float(x)), 6.0)
        # half of the gap of the interval that contains a
        k = max(j for j in range(8) if E2M1_GRID[j] <= a)
        gap = E2M1_GRID[min(k + 1, 7)] - E2M1_GRID[k] if k < 7 else 0.0
        assert abs(abs(q) - a) <= gap / 2 + 1e-12


# ------------------------------------------------------------------ E4M3
def test_e4m3_points_from_pages(orc):
    for value, code in read_golden_rows("e4m3_points.txt"):
        c = int(code, 16)
        assert orc.e4m3_encode_rne_sat(float(value)) == c
        assert orc.e4m3_decode(c) == float(value)
    # 96 = sign 0 | exponent 1101 | mantissa 100
    c = orc.e4m3_encode_rne_sat(96.0)
    assert (c >> 7, (c >> 3) & 0xF, c & 7) == (0, 0b1101, 0b100)


def test_e4m3_value_set(orc):
    vals = [orc.e4m3_decode(c) for c in range(0x7F)]
    assert len(set(vals)) == 127                      # "127 distinct sizes including zero"
    assert vals == sorted(vals)
    assert max(vals) == 448.0 and min(v for v in vals if v > 0) == 2.0 ** -9
    # eight steps inside every power of two (normal binades)
    for e in range(-6, 8):
        inside = [v for v in vals if 2.0 ** e <= v < 2.0 ** (e + 1)]
        assert len(inside) == 8 or (e == 8)


def test_e4m3_rne_ties_and_saturation(orc):
    vals = [orc.e4m3_decode(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2
        if np.float32(mid) != mid:
            continue
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode_rne_sat(mid) == want
    assert orc.e4m3_encode_rne_sat(1e9) == 0x7E
    assert orc.e4m3_encode_rne_sat(464.0) == 0x7E     # above the top midpoint: saturate
    assert orc.e4m3_encode_rne_sat(-1.0) == 0x80 | orc.e4m3_encode_rne_sat(1.0)


# ------------------------------------------------------------------ NVFP4 block scaling
def test_block_of_minus_54_gets_scale_9(orc, worked):
    ex = worked["block_neg54"]
    # s_enc = 1 exactly when the per-tensor amax is 6*448 = 2688
    s_enc, s_dec = orc.global_scales(2688.0)
    assert (s_enc, s_dec) == (1.0, 1.0)
    row = [-54.0, 5.4, 1.0, -3.0] + [0.5] * 12
    codes, scales, _, sd = orc.quantize_1d(bf16([row]), amax=2688.0)
    assert sd == 1.0
    assert orc.e4m3_decode(scales[0, 0]) == ex["scale"]
    q = unpack_codes(codes)[0]
    assert orc.e2m1_decode(q[0]) == ex["q"] and q[0] == 0xF
    # 5.4 (bf16 5.40625) / 9 -> 0.5 -> 4.5
    assert orc.e2m1_decode(q[1]) * ex["scale"] == worked["rtn_5p4"]["deq"]


def test_outer_scale_slides_the_range(orc, worked):
    r = worked["range"]
    # smallest non-zero: code 0.5 x scale 2^-9; largest: 6 x 448
    assert orc.e2m1_decode(1) * orc.e4m3_decode(0x01) == r["lo"]
    assert orc.e2m1_decode(7) * orc.e4m3_decode(0x7E) == r["hi"]
    # outer scale 2 (s_dec = 2, i.e. amax = 5376): the same block codes mean twice as much
    s_enc, s_dec = orc.global_scales(5376.0)
    assert (s_enc, s_dec) == (0.5, 2.0)
    assert orc.e2m1_decode(1) * orc.e4m3_decode(0x01) * s_dec == r["lo2"]
    assert orc.e2m1_decode(7) * orc.e4m3_decode(0x7E) * s_dec == r["hi2"]
    # a block whose max is -108 under outer scale 2 gets block scale 9 and decodes to -108
    row = [-108.0] + [1.0] * 15
    codes, scales, _, sd = orc.quantize_1d(bf16([row]), amax=5376.0)
    assert sd == 2.0 and orc.e4m3_decode(scales[0, 0]) == 9.0
    deq = orc.dequant_nvfp4(codes, scales, 1, sd)
    assert deq[0, 0] == -108.0


def test_storage_cost_bits_per_value(worked):
    n = 4096
    nvfp4_bytes = n // 2 + n // 16          # codes + one E4M3 per 16
    mxfp8_bytes = n + n // 32               # E4M3 + one E8M0 per 32
    assert nvfp4_bytes * 8 / n == worked["bits"]["nvfp4"]
    assert mxfp8_bytes * 8 / n == worked["bits"]["mxfp8"]


def test_quantize_1d_error_bound_and_block_max(orc):
    x = inputs.normal_with_outliers(64, 256, seed=11)
    xb = inputs.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    codes, scales, amax, sd = orc.quantize_1d(xb)
    assert amax == np.abs(xf).max()
    deq = orc.dequant_nvfp4(codes, scales, 1, sd)
    s = np.repeat(np.array([[orc.e4m3_decode(c) for c in r] for r in scales]), 16, axis=1) * sd
    # every element is within half of the largest E2M1 gap (2) times its block's scale,
    # or clipped at the top of the grid
    err = np.abs(deq - xf)
    assert np.all(err <= 1.0 * s + np.maximum(0, np.abs(xf) - 6 * s) + 1e-30)
    # the block max lands on the top of the grid: amax_b * s_enc_b is 6 within the
    # E4M3 rounding of the scale (a factor 1 +- 2^-4), which always rounds to 6
    dec = np.vectorize(orc.e2m1_decode)(unpack_codes(codes)).reshape(64, 16, 16)
    top = np.abs(dec).max(axis=2)
    normal = (scales > 0x01) & (scales < 0x7E)
    assert normal.any() and np.all(top[normal] == 6.0)


def test_quantize_2d_transpose_invariance(orc):
    w = inputs.normal_with_outliers(64, 96, seed=5, std=0.02)
    wb = inputs.bf16_bits(w)
    c1, s1, a1, d1 = orc.quantize_2d(wb)
    c2, s2, a2, d2 = orc.quantize_2d(np.ascontiguousarray(wb.T))
    assert a1 == a2 and d1 == d2
    assert np.array_equal(s1.T, s2)
    assert np.array_equal(unpack_codes(c1).T, unpack_codes(c2))


def test_quantize_1d_row_permutation_invariance(orc):
    x = inputs.normal_with_outliers(48, 128, seed=6)
    xb = inputs.bf16_bits(x)
    perm = np.random.default_rng(0).permutation(48)
    c1, s1, _, d1 = orc.quantize_1d(xb)
    c2, s2, _, d2 = orc.quantize_1d(np.ascontiguousarray(xb[perm]))
    assert d1 == d2
    assert np.array_equal(c1[perm], c2) and np.array_equal(s1[perm], s2)


def test_all_zero_tensor_and_underflowing_block(orc):
    z = np.zeros((16, 32), np.uint16)
    codes, scales, amax, sd = orc.quantize_1d(z)
    assert amax == 0.0 and sd == 1.0
    assert np.all(codes == 0) and np.all(scales == 0x01)
    # a block far below the tensor max: its scale would round to zero in E4M3 -> 0x01
    row = [[1e4] + [0.0] * 15 + [1e-6] * 16]
    codes, scales, _, sd = orc.quantize_1d(bf16(row))
    assert scales[0, 1] == 0x01


# ------------------------------------------------------------------ power-of-two scale
def test_pow2_ceiling_rule_worked_examples(orc, worked):
    ex = worked["pow2_22"]
    e = orc.pow2_ceil_exponent(ex["amax"], ex["vmax"])
    assert 2.0 ** e == ex["scale"]
    q = orc.e2m1_decode(orc.e2m1_encode_rne(ex["x"] / 2.0 ** e))
    assert q == ex["q"] and q * 2.0 ** e == ex["deq"]
    ex = worked["pow2_54"]
    assert 2.0 ** orc.pow2_ceil_exponent(ex["amax"], ex["vmax"]) == ex["scale"]


def test_pow2_ceiling_boundaries(orc):
    for k in (-20, -3, 0, 1, 7, 30):
        edge = 448.0 * 2.0 ** k
        assert orc.pow2_ceil_exponent(edge, 448.0) == k
        assert orc.pow2_ceil_exponent(np.nextafter(edge, np.inf), 448.0) == k + 1
        assert orc.pow2_ceil_exponent(np.nextafter(edge, 0), 448.0) == k
    assert orc.pow2_ceil_exponent(0.0, 448.0) == -127


# ------------------------------------------------------------------ Philox and SR bits
def test_philox_known_answers(orc):
    for row in read_golden_rows("philox4x32_10_kat.txt"):
        v = [int(h, 16) for h in row]
        out = orc.philox4x32_10(v[0:4], v[4:6])
        assert list(out) == v[6:10]


def test_sr_bits_counter_layout(orc):
    seed, tag = 0x0123456789ABCDEF, 3
    for blk in (0, 1, 12345, (1 << 32) + 7):
        out = orc.philox4x32_10([blk & 0xFFFFFFFF, blk >> 32, tag, 0],
                                [seed & 0xFFFFFFFF, seed >> 32])
        for j in range(8):
            w = int(out[j // 2])
            want = (w >> 16) if j % 2 else (w & 0xFFFF)
            assert orc.sr_bits16(seed, tag, blk * 8 + j) == want


def test_sr_bits_are_uniform(orc):
    r = np.array([orc.sr_bits16(7, 2, i) for i in range(40000)], dtype=np.float64)
    # mean and variance of a uniform 16-bit integer
    assert abs(r.mean() - 32767.5) < 4 * 18918.6 / math.sqrt(len(r))
    hist = np.bincount((r // 4096).astype(int), minlength=16)
    chi2 = ((hist - len(r) / 16) ** 2 / (len(r) / 16)).sum()
    assert chi2 < 45                                      # 15 dof, p ~ 1e-4


# ------------------------------------------------------------------ stochastic rounding
def test_sr_2p25_is_unbiased(orc, worked):
    ex = worked["sr_2p25"]
    n = 100000
    vals = np.array([orc.e2m1_decode(orc.e2m1_encode_sr(ex["x"], orc.sr_bits16(s, 1, 0)))
                     for s in range(n)])
    assert set(np.unique(vals)) <= {ex["lo"], ex["hi"]}
    p_hi = np.mean(vals == ex["hi"])
    sigma = math.sqrt(ex["p_hi"] * (1 - ex["p_hi"]) / n)
    assert abs(p_hi - ex["p_hi"]) < 4 * sigma
    assert abs(vals.mean() - ex["x"]) < 4 * sigma * (ex["hi"] - ex["lo"])


def test_e4m3_sr_unbiased_and_grid_fixed(orc):
    n = 100000
    rng = np.random.default_rng(1)
    for x in (0.3, 1.0 + 1 / 48, 5.1, 300.7, 2.0 ** -8 + 2.0 ** -11):
        x = float(np.float32(x))
        lo = orc.e4m3_decode(orc.e4m3_encode_rne_sat(x))
        r = rng.integers(0, 1 << 16, n)
        vals = np.array([orc.e4m3_decode(orc.e4m3_encode_sr(x, int(v))) for v in r])
        a, b = vals.min(), vals.max()
        p = (x - a) / (b - a) if b > a else 0.0
        sigma = math.sqrt(max(p * (1 - p), 1e-12) / n) * (b - a)
        assert abs(vals.mean() - x) < 4 * sigma + 2.0 ** -16 * (b - a)
        assert len(np.unique(vals)) <= 2 and a <= x <= b
        del lo
    for c in (0x01, 0x38, 0x51, 0x6C, 0x7E):   # grid values never move
        v = orc.e4m3_decode(c)
        assert all(orc.e4m3_encode_sr(v, r) == c for r in (0, 1, 32768, 65535))


def test_mxfp8_block_rne_error_bound_and_no_saturation(orc):
    rng = np.random.default_rng(3)
    for scale in (1e-3, 1.0, 700.0):
        v = (rng.standard_normal(32) * scale).astype(np.float32)
        e4, e8 = orc.mxfp8_block(v)
        e = e8 - 127
        t = np.abs(v.astype(np.float64)) / 2.0 ** e
        assert t.max() <= 448.0 and t.max() > 224.0       # ceiling rule: max lands in (224, 448]
        deq = np.array([orc.e4m3_decode(c) for c in e4]) * 2.0 ** e
        # half an E4M3 step: 2^-4 relative for normals, 2^-10 absolute in the subnormal range
        bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * 2.0 ** e)
        assert np.all(np.abs(deq - v) <= bound)


# ------------------------------------------------------------------ Hadamard
def hadamard_from_oracle(orc):
    cols = []
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        cols.append(orc.rht16_group(e, 0) * 4.0)
    return np.stack(cols, axis=1).astype(np.int64)


def test_hadamard_is_sylvester_and_orthogonal(orc):
    H = hadamard_from_oracle(orc)
    popc = np.array([[bin(i & j).count("1") for j in range(16)] for i in range(16)])
    assert np.array_equal(H, (-1) ** popc)
    assert np.array_equal(H @ H.T, 16 * np.eye(16, dtype=np.int64))


def test_rht16_inverse_and_signs(orc):
    rng = np.random.default_rng(2)
    x = rng.integers(-50, 50, 16).astype(np.float32)
    signs = 0b1010011100101101
    y = orc.rht16_group(x, signs)
    back = orc.rht16_group(y, 0)                      # (1/4 H)(1/4 H) = I
    s = np.array([-1.0 if (signs >> i) & 1 else 1.0 for i in range(16)], np.float32)
    assert np.array_equal(back * s, x)
    # definition in double: y = 1/4 H (s o x)
    H = hadamard_from_oracle(orc).astype(np.float64)
    xr = rng.standard_normal(16).astype(np.float32)
    yr = orc.rht16_group(xr, signs).astype(np.float64)
    ref = 0.25 * H @ (s * xr.astype(np.float64))
    assert np.max(np.abs(yr - ref)) <= 4 * np.finfo(np.float32).eps * np.abs(xr).sum()
    assert abs(np.linalg.norm(yr) - np.linalg.norm(xr)) <= 1e-6 * np.linalg.norm(xr)


def test_rht16_spreads_an_outlier(orc, worked):
    ex = worked["rht_outlier"]
    assert abs(ex["x"] / math.sqrt(ex["n"]) - ex["each32"]) < 0.01
    x = np.zeros(16, np.float32)
    x[5] = ex["x"]
    y = orc.rht16_group(x, 0b0110)
    assert np.all(np.abs(y) == ex["each16"])


def test_rht_cancels_in_the_wgrad_product(orc):
    """(A S H)(B S H)^T = A B^T: both wgrad operands rotated along the contraction."""
    rng = np.random.default_rng(4)
    A = rng.standard_normal((8, 64)).astype(np.float32)
    B = rng.standard_normal((5, 64)).astype(np.float32)
    signs = 0xB3C5
    RA = orc.rht16(A, signs)
    RB = orc.rht16(B, signs)
    ref = A.astype(np.float64) @ B.T.astype(np.float64)
    got = RA.astype(np.float64) @ RB.T.astype(np.float64)
    assert np.max(np.abs(got - ref)) < 1e-4 * np.abs(ref).max()
    # a wrong normalisation or a sign mismatch between operands breaks it
    RB_other = orc.rht16(B, signs ^ 1)
    bad = RA.astype(np.float64) @ RB_other.T.astype(np.float64)
    assert np.max(np.abs(bad - ref)) > 1e-2 * np.abs(ref).max()


# ------------------------------------------------------------------ requant
def test_requant_transpose_flag_equals_explicit_transpose(orc):
    dy = inputs.student_t(64, 96, seed=9)
    b = inputs.bf16_bits(dy)
    e1, s1 = orc.requant_mxfp8(orc.IN_BF16, b, None, 1.0, 64, 96, True, True, 0x1234, orc.SR, 77, 3)
    e2, s2 = orc.requant_mxfp8(orc.IN_BF16, np.ascontiguousarray(b.T), None, 1.0, 96, 64, False,
                               True, 0x1234, orc.SR, 77, 3)
    assert np.array_equal(e1, e2) and np.array_equal(s1, s2)


def test_requant_sr_is_unbiased(orc):
    """E[(w_q^T)^T] = E[w_q]: the mean over seeds of the SR requant approaches x_q."""
    w = inputs.normal(32, 64, seed=12, std=0.02)
    codes, tiles, _, sd = orc.quantize_2d(inputs.bf16_bits(w))
    xq = orc.dequant_nvfp4(codes, tiles, 2, sd)               # [32, 64]
    k = 256
    acc = np.zeros((64, 32))
    single = None
    for s in range(k):
        e4, e8 = orc.requant_mxfp8(orc.IN_NVFP4_2D, codes, tiles, sd, 32, 64, True, False, 0,
                                   orc.SR, s, 1)
        d = orc.dequant_mxfp8(e4, e8)
        acc += d
        if single is None:
            single = d
    mean = acc / k
    err1 = np.linalg.norm(single - xq.T) / np.linalg.norm(xq)
    errk = np.linalg.norm(mean - xq.T) / np.linalg.norm(xq)
    # noise averages out as 1/sqrt(k): 16x smaller for k = 256 (allow a factor 2)
    assert errk < 2 * err1 / math.sqrt(k)
    # RNE requant leaves a fixed error that averaging cannot remove
    e4, e8 = orc.requant_mxfp8(orc.IN_NVFP4_2D, codes, tiles, sd, 32, 64, True, False, 0,
                               orc.RNE, 0, 1)
    assert np.linalg.norm(orc.dequant_mxfp8(e4, e8) - xq.T) / np.linalg.norm(xq) > errk


def test_requant_nvfp4_input_matches_bf16_path_on_dequantized_values(orc):
    """NVFP4 input kinds dequantize first: feeding the same values as bf16 gives the same
    MXFP8 output whenever the dequantized values are exactly representable in bf16."""
    x = inputs.normal_with_outliers(32, 64, seed=13)
    codes, sc, _, sd = orc.quantize_1d(inputs.bf16_bits(x), amax=2688.0)   # s_dec = 1
    deq = orc.dequant_nvfp4(codes, sc, 1, sd).astype(np.float32)
    import torch
    asb = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(asb.float().numpy(), deq)                        # exact in bf16
    b = inputs.bf16_bits(asb)
    e1, s1 = orc.requant_mxfp8(orc.IN_NVFP4_1D, codes, sc, sd, 32, 64, True, True, 0xF0F0,
                               orc.SR, 5, 4)
    e2, s2 = orc.requant_mxfp8(orc.IN_BF16, b, None, 1.0, 32, 64, True, True, 0xF0F0, orc.SR, 5, 4)
    assert np.array_equal(e1, e2) and np.array_equal(s1, s2)


# ------------------------------------------------------------------ Gaussian statistics (soft)
def test_gaussian_relative_errors_match_page(orc, worked):
    ex = worked["gauss_err"]
    x = inputs.normal(256, 1024, seed=21)
    xb = inputs.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    nrm = np.linalg.norm(xf)
    codes, sc, _, sd = orc.quantize_1d(xb)
    e_nv = np.linalg.norm(orc.dequant_nvfp4(codes, sc, 1, sd) - xf) / nrm
    e4, e8 = orc.requant_mxfp8(orc.IN_BF16, xb, None, 1.0, 256, 1024, False, False, 0, orc.RNE, 0, 1)
    e_mx = np.linalg.norm(orc.dequant_mxfp8(e4, e8) - xf) / nrm
    e4, e8 = orc.requant_mxfp8(orc.IN_BF16, xb, None, 1.0, 256, 1024, False, False, 0, orc.SR, 9, 1)
    e_mx_sr = np.linalg.norm(orc.dequant_mxfp8(e4, e8) - xf) / nrm
    assert abs(e_nv / ex["nvfp4_rtn"] - 1) < 0.10, e_nv
    assert abs(e_mx / ex["mxfp8_rtn"] - 1) < 0.10, e_mx
    assert abs(e_mx_sr / ex["mxfp8_sr"] - 1) < 0.10, e_mx_sr


def test_gaussian_nvfp4_single_sr_draw_error(orc, worked):
    ex = worked["gauss_err"]
    x = inputs.normal(16, 1024, seed=22)
    xb = inputs.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    _, sc, _, sd = orc.quantize_1d(xb)
    s_enc, _ = orc.global_scales(np.abs(xf).max())
    err = 0.0
    for r in range(16):
        for b in range(64):
            enc = orc.block_encode_scale(int(sc[r, b]), sd)
            dec = orc.e4m3_decode(int(sc[r, b])) * sd
            for i in range(16):
                v = np.float32(xf[r, b * 16 + i]) * np.float32(enc)
                q = orc.e2m1_decode(orc.e2m1_encode_sr(v, orc.sr_bits16(3, 9, r * 1024 + b * 16 + i)))
                err += (q * dec - xf[r, b * 16 + i]) ** 2
    rel = math.sqrt(err) / np.linalg.norm(xf)
    assert abs(rel / ex["nvfp4_sr"] - 1) < 0.10, rel
    del s_enc


# ------------------------------------------------------------------ GEMM references
def test_gemm_special_case_exact_integers(orc):
    """Codes +-1 with every block scale 1.0 and s_dec 1: D is an exact integer matrix."""
    rng = np.random.default_rng(5)
    M, N, K = 16, 32, 64
    a = rng.choice([0x2, 0xA], size=(M, K)).astype(np.uint8)     # +1 / -1
    b = rng.choice([0x2, 0xA], size=(N, K)).astype(np.uint8)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    one = orc.e4m3_encode_rne_sat(1.0)
    D = orc.gemm_nvfp4(pack(a), np.full((M, K // 16), one, np.uint8), 1, 1.0,
                       pack(b), np.full((N // 16, K // 16), one, np.uint8), 2, 1.0)
    sa = np.where(a == 0x2, 1, -1)
    sb = np.where(b == 0x2, 1, -1)
    assert np.array_equal(D, (sa @ sb.T).astype(np.float64))


def test_gemm_nvfp4_brute_force(orc):
    """Non-square shapes, 1D x 2D scales, arbitrary s_dec: pure-Python triple loop."""
    rng = np.random.default_rng(6)
    M, N, K = 16, 48, 32
    ac = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    bc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    asc = rng.integers(0x08, 0x60, (M, K // 16), dtype=np.uint8)
    bsc = rng.integers(0x08, 0x60, (N // 16, K // 16), dtype=np.uint8)
    sa, sb = 0.375, 1.0 / 3.0
    sb = float(np.float32(sb))
    D = orc.gemm_nvfp4(ac, asc, 1, sa, bc, bsc, 2, sb)

    def code(c, r, k):
        byte = int(c[r, k // 2])
        return (byte >> 4) if k % 2 else (byte & 15)
    for m in range(M):
        for n in range(0, N, 7):
            acc = 0.0
            for k in range(K):
                va = orc.e2m1_decode(code(ac, m, k)) * orc.e4m3_decode(asc[m, k // 16]) * sa
                vb = orc.e2m1_decode(code(bc, n, k)) * orc.e4m3_decode(bsc[n // 16, k // 16]) * sb
                acc += va * vb
            assert abs(D[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_gemm_mxfp8_brute_force(orc):
    rng = np.random.default_rng(7)
    M, N, K = 3, 5, 64
    a = rng.integers(0, 0x7F, (M, K), dtype=np.uint8) | (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    b = rng.integers(0, 0x7F, (N, K), dtype=np.uint8)
    ae = rng.integers(120, 134, (M, K // 32), dtype=np.uint8)
    be = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    D = orc.gemm_mxfp8(a, ae, b, be)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += (orc.e4m3_decode(a[m, k]) * 2.0 ** (int(ae[m, k // 32]) - 127)
                        * orc.e4m3_decode(b[n, k]) * 2.0 ** (int(be[n, k // 32]) - 127))
            assert abs(D[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_round_bf16(orc):
    x = np.array([1.0, 1.00390625, 1.005859375, -3.0e-3, 65504.0], np.float32)
    import torch
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(orc.round_bf16(x), want)


# ------------------------------------------------------------------ per-row outer scale, 4/6
def test_rows_without_four_six_equal_per_tensor_quantize_of_each_row(orc):
    """With the outer scale taken per row, each row is quantized exactly as the (pinned)
    per-tensor quantizer quantizes that row on its own."""
    x = inputs.normal_with_outliers(12, 96, seed=31)
    xb = inputs.bf16_bits(x)
    codes, scales, sd = orc.quantize_1d_rows(xb, four_six=False)
    for r in range(12):
        c1, s1, _, d1 = orc.quantize_1d(xb[r:r + 1])
        assert np.array_equal(codes[r:r + 1], c1) and np.array_equal(scales[r:r + 1], s1)
        assert sd[r] == np.float32(d1)


@pytest.mark.parametrize("four_six", [False, True])
def test_rows_quantize_does_not_depend_on_other_rows(orc, four_six):
    """4bit.vizuara.ai §10: with a per-token outer scale a token's quantization does not
    depend on the other sequences in the batch. Any subset and order of rows gives the
    same bytes for each row."""
    x = inputs.normal_with_outliers(40, 128, seed=32)
    xb = inputs.bf16_bits(x)
    c, s, d = orc.quantize_1d_rows(xb, four_six)
    perm = np.random.default_rng(1).permutation(40)[:17]
    c2, s2, d2 = orc.quantize_1d_rows(np.ascontiguousarray(xb[perm]), four_six)
    assert np.array_equal(c[perm], c2) and np.array_equal(s[perm], s2) and np.array_equal(d[perm], d2)
    # a row scaled by a power of two keeps its codes and scales; its outer scale follows
    y = x.clone()
    y[3] *= 64.0
    y[5] *= 2.0 ** -20
    cy, sy, dy = orc.quantize_1d_rows(inputs.bf16_bits(y), four_six)
    assert np.array_equal(c, cy) and np.array_equal(s, sy)
    assert dy[3] == d[3] * 64 and dy[5] == np.float32(d[5] * 2.0 ** -20)
    assert np.array_equal(np.delete(d, [3, 5]), np.delete(dy, [3, 5]))


def test_four_six_worked_block(orc):
    """A block [10, 7.5, 0, ...] under outer scales 1: nothing lies between 4 and 6
    (4bit.vizuara.ai §10). Scale 10/6 rounds to the E4M3 value 1.625, 10 -> 6.15 -> 6 and
    7.5 -> 4.62 -> 4, both off; scale 10/4 = 2.5 is exact in E4M3 and stores 10 and 7.5 as
    4 and 3 exactly, so 4/6 keeps it."""
    row = [2688.0] + [0.0] * 15 + [10.0, 7.5] + [0.0] * 14        # row amax 2688: s_enc = 1
    xb = bf16([row])
    s_enc, s_dec = orc.global_scales(2688.0)
    assert s_enc == 1.0 and s_dec == 1.0
    sb6, c6, e6 = orc.nvfp4_block_candidate(xb[0, 16:], 6.0, s_enc, s_dec)
    sb4, c4, e4 = orc.nvfp4_block_candidate(xb[0, 16:], 4.0, s_enc, s_dec)
    assert orc.e4m3_decode(sb6) == 1.625 and orc.e4m3_decode(sb4) == 2.5 and sb4 == 0x42
    assert [orc.e2m1_decode(c) for c in c6[:2]] == [6.0, 4.0]
    assert [orc.e2m1_decode(c) for c in c4[:2]] == [4.0, 3.0]
    y = np.float32(10.0) * np.float32(1.0 / np.float32(1.625)), np.float32(7.5) * np.float32(1.0 / np.float32(1.625))
    want6 = ((float(y[0]) - 6) ** 2 + (float(y[1]) - 4) ** 2) * 1.625 ** 2
    assert abs(e6 - want6) <= 1e-6 * want6 and e4 == 0.0
    codes, scales, sd = orc.quantize_1d_rows(xb, four_six=True)
    assert scales[0, 1] == 0x42 and sd[0] == 1.0
    deq = orc.dequant_nvfp4_rows(codes, scales, sd)
    assert deq[0, 16] == 10.0 and deq[0, 17] == 7.5
    codes, scales, _ = orc.quantize_1d_rows(xb, four_six=False)
    assert scales[0, 1] == sb6


def test_four_six_candidate_error_is_the_scaled_squared_error(orc):
    """E_c = S_c^2 * sum (y_i - q_i)^2, recomputed here in float64 from the candidate's codes."""
    x = inputs.normal_with_outliers(1, 16 * 64, seed=33)
    xb = inputs.bf16_bits(x)[0]
    xf = x.float().numpy()[0].astype(np.float32)
    s_enc, s_dec = orc.global_scales(float(np.abs(xf).max()))
    for b in range(64):
        for target in (6.0, 4.0):
            sb, codes, err = orc.nvfp4_block_candidate(xb[16 * b:16 * b + 16], target, s_enc, s_dec)
            S = orc.e4m3_decode(sb)
            enc = np.float32(orc.block_encode_scale(sb, s_dec))
            y = (xf[16 * b:16 * b + 16] * enc).astype(np.float64)
            q = np.array([orc.e2m1_decode(int(c)) for c in codes])
            want = float(((y - q) ** 2).sum() * S * S)
            assert abs(err - want) <= 1e-5 * want + 1e-30, (b, target)
            # the error in x's own units is s_dec^2 times E_c (up to the rounding of y)
            xe = float(((xf[16 * b:16 * b + 16] - q * S * s_dec) ** 2).sum())
            assert abs(xe - want * s_dec * s_dec) <= 1e-4 * xe + 1e-30


def test_four_six_keeps_the_smaller_error_and_the_max_on_4_or_6(orc):
    """Each block keeps whichever candidate reconstructs it with the smaller squared error
    (errors recomputed in float64 from the dequantized values); with an unsaturated scale
    the block maximum sits on 6 (ordinary scale) or on 4 (the second scale)."""
    x = inputs.normal_with_outliers(16, 512, seed=34)
    xb = inputs.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    c46, s46, sd = orc.quantize_1d_rows(xb, True)
    c6, s6, sd6 = orc.quantize_1d_rows(xb, False)
    assert np.array_equal(sd, sd6)
    d46 = orc.dequant_nvfp4_rows(c46, s46, sd)
    d6 = orc.dequant_nvfp4_rows(c6, s6, sd)
    e46 = ((d46 - xf) ** 2).reshape(16, 32, 16).sum(-1)
    e6 = ((d6 - xf) ** 2).reshape(16, 32, 16).sum(-1)
    changed = s46 != s6
    assert changed.any() and (~changed).any()
    assert np.all(e46 <= e6 * (1 + 1e-5) + 1e-30)
    assert np.all(e46[changed] < e6[changed])
    # every changed block used the 4 candidate: its scale is the one for target 4
    amax_b = np.abs(xf).reshape(16, 32, 16).max(-1)
    for r, b in zip(*np.nonzero(changed)):
        s_enc = orc.global_scales(float(np.abs(xf[r]).max()))[0]
        assert s46[r, b] == orc.nvfp4_block_candidate(xb[r, 16 * b:16 * b + 16], 4.0, s_enc, sd[r])[0]
    top = np.abs(np.vectorize(orc.e2m1_decode)(unpack_codes(c46))).reshape(16, 32, 16).max(-1)
    normal = (s46 > 0x08) & (s46 < 0x70)
    assert np.all(top[normal & changed] == 4.0) and np.all(top[normal & ~changed] == 6.0)
    assert np.all(amax_b[normal] > 0)


def test_four_six_lowers_the_error_like_the_page(orc, worked):
    """4bit.vizuara.ai §10 reports 9.3% -> 8.9% (MLP input) and 8.3% -> 8.1% (after GELU) on
    real activations; on synthetic Gaussian and GELU-of-Gaussian inputs the relative error
    drops by a similar few percent."""
    import torch
    ex = worked["four_six"]
    lo = min(ex["in_46"] / ex["in_6"], ex["gelu_46"] / ex["gelu_6"]) - 0.05
    for x in (inputs.normal(128, 1024, seed=35),
              torch.nn.functional.gelu(inputs.normal(128, 1024, seed=36).float()).to(torch.bfloat16)):
        xb = inputs.bf16_bits(x)
        xf = x.float().numpy().astype(np.float64)
        n = np.linalg.norm(xf)
        e = []
        for fs in (False, True):
            c, s, sd = orc.quantize_1d_rows(xb, fs)
            e.append(np.linalg.norm(orc.dequant_nvfp4_rows(c, s, sd) - xf) / n)
        assert lo < e[1] / e[0] < 1.0, e


def test_rows_all_zero_row_and_tiny_row(orc):
    codes, scales, sd = orc.quantize_1d_rows(bf16([[0.0] * 32, [1e-30] + [0.0] * 31]), True)
    assert sd[0] == 1.0 and np.all(scales[0] == 0x01) and np.all(codes[0] == 0)
    # a lone tiny value is its row's max: its block scale is 448 and it is stored as 6
    v = float(np.array([int(bf16([1e-30])[0]) << 16], np.uint32).view(np.float32)[0])
    assert scales[1, 0] == 0x7E and (codes[1, 0] & 0x0F) == 0x7
    deq = orc.dequant_nvfp4_rows(codes, scales, sd)
    assert abs(deq[1, 0] - v) <= 1e-6 * v and np.all(deq[1, 1:] == 0)


def test_requant_per_row_outer_scale_input(orc):
    """Input kind 3 dequantizes with each row's own outer scale. With power-of-two outer
    scales the dequantized values are exact in bf16, so the result equals the bf16 path on
    those values; with equal outer scales it equals kind 1."""
    import torch
    x = inputs.normal_with_outliers(64, 64, seed=37)
    x = x.float() * (2.0 ** torch.arange(-8, 8).repeat(4))[:, None]
    x[:, 0] = 2688.0 * (2.0 ** torch.arange(-8, 8).repeat(4))          # row amax 2688 * 2^k
    xb = inputs.bf16_bits(x.to(torch.bfloat16))
    codes, sc, sd = orc.quantize_1d_rows(xb, True)
    assert np.array_equal(sd, (2.0 ** np.arange(-8, 8)).repeat(1).astype(np.float32)[np.arange(64) % 16])
    deq = orc.dequant_nvfp4_rows(codes, sc, sd).astype(np.float32)
    asb = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(asb.float().numpy(), deq)
    for tr, rht, rnd in ((True, True, orc.SR), (False, False, orc.RNE), (True, False, orc.SR)):
        e1, s1 = orc.requant_mxfp8(orc.IN_NVFP4_1D_ROWS, codes, sc, sd, 64, 64, tr, rht, 0x1234, rnd, 3, 2)
        e2, s2 = orc.requant_mxfp8(orc.IN_BF16, inputs.bf16_bits(asb), None, 1.0, 64, 64, tr, rht, 0x1234,
                                   rnd, 3, 2)
        assert np.array_equal(e1, e2) and np.array_equal(s1, s2)
    c1, s1d, _, d1 = orc.quantize_1d(xb[:1])
    same = np.full(64, np.float32(d1), np.float32)
    e1, s1 = orc.requant_mxfp8(orc.IN_NVFP4_1D_ROWS, codes, sc, same, 64, 64, True, True, 7, orc.SR, 1, 1)
    e2, s2 = orc.requant_mxfp8(orc.IN_NVFP4_1D, codes, sc, float(d1), 64, 64, True, True, 7, orc.SR, 1, 1)
    assert np.array_equal(e1, e2) and np.array_equal(s1, s2)


def test_gemm_nvfp4_rows_brute_force(orc):
    """A carries one outer scale per row: pure-Python triple loop on tiny shapes."""
    rng = np.random.default_rng(8)
    M, N, K = 8, 16, 32
    ac = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    bc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    asc = rng.integers(0x08, 0x60, (M, K // 16), dtype=np.uint8)
    bsc = rng.integers(0x08, 0x60, (N // 16, K // 16), dtype=np.uint8)
    sa = rng.uniform(0.1, 3.0, M).astype(np.float32)
    sb = float(np.float32(0.7))
    D = orc.gemm_nvfp4_rows(ac, asc, sa, bc, bsc, 2, sb)

    def code(c, r, k):
        byte = int(c[r, k // 2])
        return (byte >> 4) if k % 2 else (byte & 15)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                va = orc.e2m1_decode(code(ac, m, k)) * orc.e4m3_decode(asc[m, k // 16]) * float(sa[m])
                vb = orc.e2m1_decode(code(bc, n, k)) * orc.e4m3_decode(bsc[n // 16, k // 16]) * sb
                acc += va * vb
            assert abs(D[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


# ------------------------------------------------------------------ combine codec: RHT32 + S2F6
def test_s2f6_grid_matches_page(orc, worked):
    ex = worked["s2f6"]
    vals = sorted(orc.s2f6_decode(c, 127) for c in range(256))        # E8M0 127: scale 1
    assert vals[0] == ex["lo"] and vals[-1] == ex["hi"]
    assert np.allclose(np.diff(vals), ex["step"], rtol=0, atol=0)
    assert (8 * 32 + 8) / 32 == ex["bits"]
    # the scale is a plain power of two
    assert orc.s2f6_decode(64, 130) == 8.0 and orc.s2f6_decode(0x80, 120) == -2.0 * 2.0 ** -7


def test_rht32_is_the_normalised_sylvester_hadamard(orc):
    c = float(np.float32(0.17677669529663688))             # RN(1/sqrt(32))
    for signs in (0, 0x8000_0001, 0x5A5A_C3C3):
        cols = []
        for j in range(32):
            e = np.zeros(32, np.float32)
            e[j] = 1.0
            cols.append(orc.rht32_group(e, signs))
        H = np.array(cols).T
        i = np.arange(32)
        want = np.array([[(-1) ** bin(a & b).count("1") for b in i] for a in i], np.float64)
        s = np.array([-1.0 if (signs >> k) & 1 else 1.0 for k in range(32)])
        assert np.array_equal(H, (want * s[None, :] * c).astype(np.float32))
        assert np.allclose(H @ H.T, np.eye(32), atol=1e-6)


def test_rht32_inverse_energy_and_outlier_spread(orc, worked):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(32).astype(np.float32)
    signs = 0x1234_ABCD
    y = orc.rht32_group(x, signs)
    assert abs(np.linalg.norm(y) / np.linalg.norm(x) - 1) < 1e-6
    assert np.allclose(orc.irht32_group(y, signs), x, rtol=0, atol=1e-6)
    spike = np.zeros(32, np.float32)
    spike[7] = worked["rht_outlier"]["x"]
    out = orc.rht32_group(spike, signs)
    assert np.allclose(np.abs(out), worked["rht_outlier"]["each32"], atol=0.01)


def test_s2f6_scale_rule_rounding_and_saturation(orc):
    # the block max decides: amax <= (127/64) 2^e for the smallest e
    for k in (-3, 0, 5):
        y = np.zeros(32, np.float32)
        y[0] = 127 / 64 * 2.0 ** k
        codes, e8 = orc.s2f6_block(y)
        assert e8 == 127 + k and np.int8(codes[0]) == 127
        y[0] = np.nextafter(np.float32(y[0]), np.float32(np.inf))
        codes, e8 = orc.s2f6_block(y)
        assert e8 == 128 + k
    zero_codes, zero_e8 = orc.s2f6_block(np.zeros(32, np.float32))
    assert zero_e8 == 0 and not zero_codes.any()
    # ties to even in units of 1/64 of the scale (block max 1.5 -> e = 0)
    y = np.zeros(32, np.float32)
    y[:6] = [1.5, 2.5 / 64, 3.5 / 64, -2.5 / 64, -0.5 / 64, 0.5 / 64]
    codes, e8 = orc.s2f6_block(y)
    assert e8 == 127
    assert [int(np.int8(c)) for c in codes[:6]] == [96, 2, 4, -2, 0, 0]
    # negative values use the full range down to -2 only when the positive side allows it
    y[:] = -1.0
    codes, e8 = orc.s2f6_block(y)
    assert e8 == 127 and np.all(codes.view(np.int8) == -64)


def test_combine_decode_sums_arrivals_then_rotates_back(orc):
    rng = np.random.default_rng(4)
    signs = 0x0F0F_3C3C
    k, tokens, cols = 3, 5, 64
    x = rng.standard_normal((tokens * k, cols)).astype(np.float32) * 3
    codes, e8 = orc.combine_encode(x, signs)
    out = orc.combine_decode(codes, e8, k, signs)
    for t in range(tokens):
        for g in range(cols // 32):
            acc = None
            for j in range(k):
                r = t * k + j
                z = np.array([orc.s2f6_decode(c, e8[r, g]) for c in codes[r, 32 * g:32 * g + 32]], np.float32)
                acc = z if acc is None else (acc + z).astype(np.float32)
            assert np.array_equal(out[t, 32 * g:32 * g + 32], orc.irht32_group(acc, signs))
    # and it approximates the sum of the inputs
    ref = x.reshape(tokens, k, cols).sum(axis=1)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 0.02


def test_combine_round_trip_within_half_a_step(orc):
    """One arrival: each value's rotated-domain error is at most half a step 2^(e-7); the
    rotation back is orthonormal, so each group's error norm is at most sqrt(32) 2^(e-7)."""
    x = inputs.student_t(16, 256, seed=5, df=3, scale=1.0).float().numpy()
    signs = 0xDEAD_BEEF
    codes, e8 = orc.combine_encode(x, signs)
    out = orc.combine_decode(codes, e8, 1, signs)
    err = np.linalg.norm((out - x).reshape(16, 8, 32), axis=2)
    bound = np.sqrt(32) * 2.0 ** (e8.astype(np.float64) - 127 - 7)
    assert np.all(err <= bound * (1 + 1e-5) + 1e-5 * np.linalg.norm(x.reshape(16, 8, 32), axis=2))


def test_wire_format_errors_order_like_page(orc, worked):
    """4bit.vizuara.ai §11 on real MLP outputs: MXFP8 2.66% > S2F6 0.92% > RHT32 + S2F6 0.79%, and
    the rotation lowers the kurtosis (59 -> 7) and the spikiest block (5.6x -> 1.3x). The same
    ordering holds on heavy-tailed synthetic outputs (Student-t, 3 degrees of freedom)."""
    ex = worked["wire"]
    x = inputs.student_t(64, 1024, seed=6, df=3, scale=1.0).float().numpy()
    xb = np.ascontiguousarray(x.astype(np.float32))
    n = np.linalg.norm(xb)
    e4, e8 = orc.requant_mxfp8(orc.IN_BF16, inputs.bf16_bits(inputs.student_t(64, 1024, seed=6, df=3, scale=1.0)),
                               None, 1.0, 64, 1024, False, False, 0, orc.RNE, 0, 1)
    e_mx = np.linalg.norm(orc.dequant_mxfp8(e4, e8) - xb) / n
    # S2F6 without the rotation: quantize the raw blocks
    raw = np.zeros_like(xb)
    for r in range(64):
        for g in range(32):
            cc, ee = orc.s2f6_block(xb[r, 32 * g:32 * g + 32])
            raw[r, 32 * g:32 * g + 32] = [orc.s2f6_decode(q, ee) for q in cc]
    e_s2f6 = np.linalg.norm(raw - xb) / n
    signs = 0x9E37_79B9
    c, s = orc.combine_encode(xb, signs)
    e_rht = np.linalg.norm(orc.combine_decode(c, s, 1, signs) - xb) / n
    assert e_mx > e_s2f6 > e_rht, (e_mx, e_s2f6, e_rht)
    assert e_mx / e_s2f6 > 0.5 * ex["mxfp8"] / ex["s2f6"]
    blocks = xb.reshape(-1, 32)
    rot = np.array([orc.rht32_group(b, signs) for b in blocks])
    kurt = lambda v: float(np.mean(v ** 4) / np.mean(v ** 2) ** 2)
    assert kurt(rot) < kurt(blocks) / 2 and kurt(rot) < ex["kurt"]
    spike = lambda b: float(np.max(np.abs(b)) / np.sqrt(np.mean(b ** 2)))
    worst = int(np.argmax([spike(b) for b in blocks]))
    assert spike(rot[worst]) < spike(blocks[worst]) / 2


# ------------------------------------------------------------------ MXFP4 (the format comparison)
def test_mxfp4_worked_examples(orc, worked):
    """[AC] "The scaling math, worked": amax 22 -> scale 2^ceil(log2(22/6)) = 4, 22 -> 5.5 -> 6 -> 24.
    [NV] App. B.4: a block with amax 3 + delta keeps 3 as its largest code (power-of-two scale 1),
    while amax exactly 3 gets scale 1/2 and reaches 6."""
    ex = worked["pow2_22"]
    row = [ex["x"]] + [0.0] * 31
    codes, e8 = orc.quantize_mxfp4(bf16([row]))
    assert 2.0 ** (int(e8[0, 0]) - 127) == ex["scale"]
    assert orc.dequant_mxfp4(codes, e8)[0, 0] == ex["deq"]
    codes, e8 = orc.quantize_mxfp4(bf16([[3.015625] + [0.0] * 31]))
    assert e8[0, 0] == 127 and orc.dequant_mxfp4(codes, e8)[0, 0] == 3.0
    codes, e8 = orc.quantize_mxfp4(bf16([[3.0] + [0.0] * 31]))
    assert e8[0, 0] == 126 and (codes[0, 0] & 0x7) == 0x7
    # a block max of exactly 6 * 2^k keeps scale 2^k and the top code
    for k in (-20, 0, 9):
        codes, e8 = orc.quantize_mxfp4(bf16([[6.0 * 2.0 ** k] + [0.0] * 31]))
        assert e8[0, 0] == 127 + k and (codes[0, 0] & 0x7) == 0x7


def test_mxfp4_gemm_brute_force(orc):
    rng = np.random.default_rng(11)
    M, N, K = 5, 7, 64
    ac = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    bc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ae = rng.integers(118, 136, (M, K // 32), dtype=np.uint8)
    be = rng.integers(118, 136, (N, K // 32), dtype=np.uint8)
    D = orc.gemm_mxfp4(ac, ae, bc, be)

    def code(c, r, k):
        byte = int(c[r, k // 2])
        return (byte >> 4) if k % 2 else (byte & 15)
    for m in range(M):
        for n in range(N):
            acc = sum(orc.e2m1_decode(code(ac, m, k)) * 2.0 ** (int(ae[m, k // 32]) - 127)
                      * orc.e2m1_decode(code(bc, n, k)) * 2.0 ** (int(be[n, k // 32]) - 127) for k in range(K))
            assert abs(D[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_mxfp4_error_above_nvfp4_and_rht_on_heavy_tails(orc):
    """The pages' format comparison: power-of-two scales per 32 lose accuracy against E4M3
    scales per 16 ([NV] "NVFP4 vs. MXFP4"; [AC] micro-scaling). With a 32-point rotation first,
    MXFP4's error on heavy-tailed data drops ([NV] Section 5 pairs MXFP4 with d = 32)."""
    x = inputs.normal(64, 1024, seed=41)
    xb = inputs.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    n = np.linalg.norm(xf)
    c, e = orc.quantize_mxfp4(xb)
    e_mx = np.linalg.norm(orc.dequant_mxfp4(c, e) - xf) / n
    c1, s1, _, sd = orc.quantize_1d(xb)
    e_nv = np.linalg.norm(orc.dequant_nvfp4(c1, s1, 1, sd) - xf) / n
    assert 0.08 < e_nv < e_mx < 0.14, (e_nv, e_mx)
    t = inputs.student_t(32, 1024, seed=42, df=3, scale=1.0)
    tb = inputs.bf16_bits(t)
    tf = t.float().numpy().astype(np.float32)
    signs = 0x5EED_1234
    c, e = orc.quantize_mxfp4(tb)
    e_plain = np.linalg.norm(orc.dequant_mxfp4(c, e) - tf) / np.linalg.norm(tf)
    c, e = orc.quantize_mxfp4(tb, rht=True, signs=signs)
    rot = np.array([orc.rht32_group(b, signs) for b in tf.reshape(-1, 32)]).reshape(tf.shape)
    e_rht = np.linalg.norm(orc.dequant_mxfp4(c, e) - rot) / np.linalg.norm(rot)
    assert e_rht < e_plain, (e_rht, e_plain)
    # with the rotation, a block is the plain MXFP4 rule applied to the rotated values
    codes, e8 = orc.quantize_mxfp4(tb[:1], rht=True, signs=signs)
    v = orc.rht32_group(tf[0, :32], signs)
    sc = 2.0 ** (int(e8[0, 0]) - 127)
    assert sc == 2.0 ** orc.pow2_ceil_exponent(float(np.abs(v).max()), 6.0)
    want = [orc.e2m1_encode_rne(np.float32(vi / sc)) for vi in v]
    assert [int(c) for c in unpack_codes(codes)[0, :32]] == want


# ---------------------------------------------------------------- GELU (4bit.vizuara.ai §13-14)
def test_normal_cdf_and_erfc_against_printed_tables(orc):
    """Phi and erfc at the points printed in standard tables (tests/golden/normal_cdf.txt),
    including the far lower tail, where Phi computed as (1 + erf)/2 would cancel to zero."""
    for kind, x, v in read_golden_rows("normal_cdf.txt"):
        x, v = float(x), float(v)
        got = orc.normal_cdf(x) if kind == "phi" else 2.0 * orc.normal_cdf(-x * math.sqrt(2.0))
        assert abs(got - v) <= 1e-13 * abs(v), (kind, x, got, v)


def test_gelu_closed_forms(orc):
    """GELU(0) = 0 and GELU'(0) = Phi(0) = 1/2; GELU(x) - GELU(-x) = x (Phi(x) + Phi(-x) = 1);
    GELU'(x) + GELU'(-x) = 1; GELU(x) -> x above and -> 0 below, with the tail value
    x Phi(x) at -10 from the table."""
    assert orc.gelu(0.0) == 0.0 and orc.gelu_grad(0.0) == 0.5
    for x in np.linspace(-9.0, 9.0, 181):
        x = float(x)
        assert abs(orc.gelu(x) - orc.gelu(-x) - x) <= 1e-15 * max(1.0, abs(x))
        assert abs(orc.gelu_grad(x) + orc.gelu_grad(-x) - 1.0) <= 1e-15
    assert orc.gelu(10.0) == 10.0
    assert abs(orc.gelu(-10.0) - (-10.0 * 7.61985302416052e-24)) <= 1e-13 * 7.62e-23
    # the page's examples of the activation are bf16 tensors: the batch form agrees
    h = inputs.bf16_bits(inputs.normal(4, 64, seed=5, std=3.0))
    hv = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(orc.gelu_bf16(h), np.vectorize(orc.gelu)(hv))
    assert np.array_equal(orc.gelu_bf16(h, grad=True), np.vectorize(orc.gelu_grad)(hv))


def test_gelu_grad_is_the_derivative_of_gelu(orc):
    """GELU' against a central difference of the oracle's own GELU (step 1e-5: truncation
    error ~1e-11, rounding ~1e-11): a dropped term or a wrong sign in x phi(x) fails."""
    d = 1e-5
    for x in np.linspace(-8.0, 8.0, 321):
        x = float(x)
        fd = (orc.gelu(x + d) - orc.gelu(x - d)) / (2 * d)
        assert abs(fd - orc.gelu_grad(x)) <= 1e-8, (x, fd, orc.gelu_grad(x))
    # the density: phi(0) = 1/sqrt(2 pi), and phi integrates Phi (one Simpson panel check)
    assert abs(orc.normal_pdf(0.0) - 0.3989422804014327) <= 1e-16
    xs = np.linspace(-1.0, 1.0, 2001)
    ys = np.array([orc.normal_pdf(float(v)) for v in xs])
    simpson = (xs[1] - xs[0]) / 3 * (ys[0] + ys[-1] + 4 * ys[1:-1:2].sum() + 2 * ys[2:-1:2].sum())
    assert abs(simpson - (orc.normal_cdf(1.0) - orc.normal_cdf(-1.0))) <= 1e-12
