"""numpy-level API over the C oracle (``fp4q_oracle.c``).

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of the benchmark).

bf16 tensors are passed as ``np.uint16`` bit patterns. Packed NVFP4 codes are
``[rows, cols/2]`` bytes with element ``2j`` in the low nibble; NVFP4 scales are
E4M3 bytes, ``[rows, cols/16]`` (1D) or ``[rows/16, cols/16]`` (16x16 tiles);
MXFP8 is E4M3 bytes ``[rows, cols]`` plus E8M0 bytes ``[rows, cols/32]``.

The GEMM references dequantize each operand exactly (in float64) and multiply with
a float64 matmul: the block-scaled GEMM of the pages ("Pretraining Large Language
Models with NVFP4", Quantization Procedure step 5; 4bit.vizuara.ai §7) is, up to the
order of its fp32 additions, exactly this product.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64

RNE, SR = 0, 1
IN_BF16, IN_NVFP4_1D, IN_NVFP4_2D, IN_NVFP4_1D_ROWS = 0, 1, 2, 3


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint32]
        L.orc_e2m1_encode_rne.restype = ctypes.c_uint32
        L.orc_e2m1_encode_rne.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode_sr.restype = ctypes.c_uint32
        L.orc_e2m1_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint32]
        L.orc_e4m3_encode_rne_sat.restype = ctypes.c_uint32
        L.orc_e4m3_encode_rne_sat.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode_sr.restype = ctypes.c_uint32
        L.orc_e4m3_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.orc_pow2_ceil_exponent.restype = ctypes.c_int
        L.orc_pow2_ceil_exponent.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_philox4x32_10.restype = None
        L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.orc_sr_bits16.restype = ctypes.c_uint32
        L.orc_sr_bits16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        L.orc_amax_bf16.restype = ctypes.c_float
        L.orc_amax_bf16.argtypes = [_u16p, _i64, _i64, _i64]
        L.orc_global_scales.restype = None
        L.orc_global_scales.argtypes = [ctypes.c_float, _f32p, _f32p]
        L.orc_block_scale_code.restype = ctypes.c_uint32
        L.orc_block_scale_code.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_block_encode_scale.restype = ctypes.c_float
        L.orc_block_encode_scale.argtypes = [ctypes.c_uint32, ctypes.c_float]
        for fn in (L.orc_quantize_1d, L.orc_quantize_2d):
            fn.restype = None
            fn.argtypes = [_u16p, _i64, _i64, _i64, _f32p, _u8p, _u8p, _f32p, _f32p]
        L.orc_nvfp4_block_candidate.restype = None
        L.orc_nvfp4_block_candidate.argtypes = [_u16p, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                _u32p, _u8p, _f32p]
        L.orc_quantize_1d_rows.restype = None
        L.orc_quantize_1d_rows.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_int, _u8p, _u8p, _f32p]
        L.orc_dequant_nvfp4_rows.restype = None
        L.orc_dequant_nvfp4_rows.argtypes = [_u8p, _u8p, _f32p, _i64, _i64, _f32p, _f64p]
        L.orc_dequant_nvfp4.restype = None
        L.orc_dequant_nvfp4.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_float, _i64, _i64,
                                        _f32p, _f64p]
        L.orc_dequant_mxfp8.restype = None
        L.orc_dequant_mxfp8.argtypes = [_u8p, _u8p, _i64, _i64, _f64p]
        L.orc_rht16_group.restype = None
        L.orc_rht16_group.argtypes = [_f32p, ctypes.c_uint32]
        L.orc_rht16.restype = None
        L.orc_rht16.argtypes = [ctypes.c_void_p, ctypes.c_int, _f32p, _i64, _i64, ctypes.c_uint32]
        L.orc_mxfp8_block.restype = None
        L.orc_mxfp8_block.argtypes = [_f32p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32,
                                      ctypes.c_uint64, _u8p, _u8p]
        L.orc_requant_mxfp8_rows.restype = None
        L.orc_requant_mxfp8_rows.argtypes = [ctypes.c_int, ctypes.c_void_p, _u8p, ctypes.c_float,
                                             _f32p, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                             ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32, _i64, _i64,
                                             _u8p, _u8p]
        L.orc_requant_mxfp8.restype = None
        L.orc_requant_mxfp8.argtypes = [ctypes.c_int, ctypes.c_void_p, _u8p, ctypes.c_float,
                                        _f32p, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                        ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32, _u8p, _u8p]
        L.orc_rht32_group.restype = None
        L.orc_rht32_group.argtypes = [_f32p, ctypes.c_uint32]
        L.orc_irht32_group.restype = None
        L.orc_irht32_group.argtypes = [_f32p, ctypes.c_uint32]
        L.orc_s2f6_block.restype = None
        L.orc_s2f6_block.argtypes = [_f32p, _u8p, _u8p]
        L.orc_s2f6_decode.restype = ctypes.c_double
        L.orc_s2f6_decode.argtypes = [ctypes.c_uint8, ctypes.c_uint8]
        L.orc_combine_encode.restype = None
        L.orc_combine_encode.argtypes = [ctypes.c_void_p, ctypes.c_int, _i64, _i64, ctypes.c_uint32, _u8p, _u8p]
        L.orc_combine_decode.restype = None
        L.orc_combine_decode.argtypes = [_u8p, _u8p, _i64, _i64, _i64, ctypes.c_uint32, _f32p]
        L.orc_quantize_mxfp4.restype = None
        L.orc_quantize_mxfp4.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_int, ctypes.c_uint32, _u8p, _u8p]
        L.orc_dequant_mxfp4.restype = None
        L.orc_dequant_mxfp4.argtypes = [_u8p, _u8p, _i64, _i64, _f64p]
        for fn in (L.orc_normal_cdf, L.orc_normal_pdf, L.orc_gelu, L.orc_gelu_grad):
            fn.restype = ctypes.c_double
            fn.argtypes = [ctypes.c_double]
        L.orc_gelu_bf16.restype = None
        L.orc_gelu_bf16.argtypes = [_u16p, _i64, ctypes.c_int, _f64p]
        _LIB = L
    return _LIB


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def e2m1_decode(code):
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode_rne(v):
    return lib().orc_e2m1_encode_rne(float(v))


def e2m1_encode_sr(v, r16):
    return lib().orc_e2m1_encode_sr(float(v), int(r16))


def e4m3_decode(code):
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode_rne_sat(v):
    return lib().orc_e4m3_encode_rne_sat(float(v))


def e4m3_encode_sr(v, r16):
    return lib().orc_e4m3_encode_sr(float(v), int(r16))


def pow2_ceil_exponent(amax, vmax):
    return lib().orc_pow2_ceil_exponent(float(amax), float(vmax))


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def sr_bits16(seed, tag, idx):
    return lib().orc_sr_bits16(int(seed), int(tag), int(idx))


def global_scales(amax):
    e = ctypes.c_float()
    d = ctypes.c_float()
    lib().orc_global_scales(float(amax), ctypes.byref(e), ctypes.byref(d))
    return e.value, d.value


def block_scale_code(amax_b, s_enc):
    return lib().orc_block_scale_code(float(amax_b), float(s_enc))


def block_encode_scale(sb, s_dec):
    return lib().orc_block_encode_scale(int(sb), float(s_dec))


# ---------------------------------------------------------------- tensors
def amax_bf16(x):
    x = _c(x, np.uint16)
    return lib().orc_amax_bf16(_p(x, _u16p), x.shape[0], x.shape[1], x.shape[1])


def _quantize(fn, x, amax, tile):
    x = _c(x, np.uint16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows // 16, cols // 16) if tile else (rows, cols // 16), np.uint8)
    a_in = None if amax is None else ctypes.byref(ctypes.c_float(amax))
    a_out = ctypes.c_float()
    s_dec = ctypes.c_float()
    fn(_p(x, _u16p), rows, cols, cols, a_in, _p(codes, _u8p), _p(scales, _u8p),
       ctypes.byref(a_out), ctypes.byref(s_dec))
    return codes, scales, a_out.value, s_dec.value


def quantize_1d(x, amax=None):
    """NVFP4 with 1x16 blocks along rows -> (codes, scales, amax, s_dec)."""
    return _quantize(lib().orc_quantize_1d, x, amax, tile=False)


def quantize_2d(w, amax=None):
    """NVFP4 with 16x16 tile scales -> (codes, tile_scales, amax, s_dec)."""
    return _quantize(lib().orc_quantize_2d, w, amax, tile=True)


def nvfp4_block_candidate(xb, target, s_enc, s_dec):
    """One 4/6 candidate for 16 bf16 values (uint16 bits), target 6.0 or 4.0
    -> (scale code, codes[16], error E_c)."""
    xb = _c(xb, np.uint16)
    assert xb.size == 16
    sb = ctypes.c_uint32()
    codes = np.zeros(16, np.uint8)
    err = ctypes.c_float()
    lib().orc_nvfp4_block_candidate(_p(xb, _u16p), float(target), float(s_enc), float(s_dec),
                                    ctypes.byref(sb), _p(codes, _u8p), ctypes.byref(err))
    return sb.value, codes, err.value


def quantize_1d_rows(x, four_six=True):
    """NVFP4 1x16 blocks with a per-row outer scale (and 4/6 if four_six)
    -> (codes, scales, s_dec_rows float32[rows])."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    s_dec = np.zeros(rows, np.float32)
    lib().orc_quantize_1d_rows(_p(x, _u16p), rows, cols, cols, int(bool(four_six)),
                               _p(codes, _u8p), _p(scales, _u8p), _p(s_dec, _f32p))
    return codes, scales, s_dec


def dequant_nvfp4_rows(codes, scales, s_dec_rows, as_f32=False):
    """1D scales with a per-row outer scale s_dec_rows[rows]."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    sd = _c(s_dec_rows, np.float32)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float32 if as_f32 else np.float64)
    lib().orc_dequant_nvfp4_rows(_p(codes, _u8p), _p(scales, _u8p), _p(sd, _f32p), rows, cols,
                                 _p(out, _f32p) if as_f32 else None,
                                 None if as_f32 else _p(out, _f64p))
    return out


def dequant_nvfp4(codes, scales, scale_kind, s_dec, as_f32=False):
    """scale_kind 1 = 1D [rows, cols/16], 2 = tiles [rows/16, cols/16]."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    if as_f32:
        out = np.zeros((rows, cols), np.float32)
        lib().orc_dequant_nvfp4(_p(codes, _u8p), _p(scales, _u8p), scale_kind, float(s_dec),
                                rows, cols, _p(out, _f32p), None)
    else:
        out = np.zeros((rows, cols), np.float64)
        lib().orc_dequant_nvfp4(_p(codes, _u8p), _p(scales, _u8p), scale_kind, float(s_dec),
                                rows, cols, None, _p(out, _f64p))
    return out


def dequant_mxfp8(e4m3, e8m0):
    e4m3 = _c(e4m3, np.uint8)
    e8m0 = _c(e8m0, np.uint8)
    rows, cols = e4m3.shape
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_mxfp8(_p(e4m3, _u8p), _p(e8m0, _u8p), rows, cols, _p(out, _f64p))
    return out


def rht16_group(v, signs):
    v = _c(v, np.float32).copy()
    lib().orc_rht16_group(_p(v, _f32p), int(signs))
    return v


def rht16(x, signs, is_bf16=False):
    x = _c(x, np.uint16 if is_bf16 else np.float32)
    rows, cols = x.shape
    out = np.zeros((rows, cols), np.float32)
    lib().orc_rht16(x.ctypes.data, int(bool(is_bf16)), _p(out, _f32p), rows, cols, int(signs))
    return out


def mxfp8_block(v, rounding=RNE, seed=0, tag=0, out_idx0=0):
    v = _c(v, np.float32)
    e4 = np.zeros(32, np.uint8)
    e8 = np.zeros(1, np.uint8)
    lib().orc_mxfp8_block(_p(v, _f32p), rounding, int(seed), int(tag), int(out_idx0),
                          _p(e4, _u8p), _p(e8, _u8p))
    return e4, int(e8[0])


def requant_mxfp8(in_kind, data, scales, s_dec, rows, cols, transpose, rht, rht_signs,
                  rounding, seed, tag, out_rows=None):
    """Dequantize -> [transpose] -> [RHT16] -> MXFP8 -> (e4m3, e8m0).
    in_kind IN_NVFP4_1D_ROWS takes s_dec as an array of per-row outer scales.
    out_rows=(begin, end) computes only those output rows."""
    sd_rows = None
    if in_kind == IN_NVFP4_1D_ROWS:
        sd_rows = _c(s_dec, np.float32)
        assert sd_rows.shape == (rows,)
        s_dec = 0.0
    if in_kind == IN_BF16:
        data = _c(data, np.uint16)
        sc = None
    else:
        data = _c(data, np.uint8)
        scales = _c(scales, np.uint8)
        sc = _p(scales, _u8p)
    orows, ocols = (cols, rows) if transpose else (rows, cols)
    b, e = (0, orows) if out_rows is None else out_rows
    e4 = np.zeros((e - b, ocols), np.uint8)
    e8 = np.zeros((e - b, ocols // 32), np.uint8)
    lib().orc_requant_mxfp8_rows(in_kind, data.ctypes.data, sc, float(s_dec),
                                 None if sd_rows is None else _p(sd_rows, _f32p), rows, cols,
                                 int(bool(transpose)), int(bool(rht)), int(rht_signs), rounding,
                                 int(seed), int(tag), b, e, _p(e4, _u8p), _p(e8, _u8p))
    return e4, e8


# ---------------------------------------------------------------- combine codec (RHT32 + S2F6)
def rht32_group(v, signs):
    v = _c(v, np.float32).copy()
    assert v.size == 32
    lib().orc_rht32_group(_p(v, _f32p), int(signs))
    return v


def irht32_group(v, signs):
    v = _c(v, np.float32).copy()
    assert v.size == 32
    lib().orc_irht32_group(_p(v, _f32p), int(signs))
    return v


def s2f6_block(y):
    """32 fp32 values -> (codes uint8[32] two's complement, e8m0 byte)."""
    y = _c(y, np.float32)
    codes = np.zeros(32, np.uint8)
    e8 = np.zeros(1, np.uint8)
    lib().orc_s2f6_block(_p(y, _f32p), _p(codes, _u8p), _p(e8, _u8p))
    return codes, int(e8[0])


def s2f6_decode(code, e8m0):
    return lib().orc_s2f6_decode(int(code) & 0xFF, int(e8m0))


def combine_encode(x, signs, is_bf16=False):
    """[rows, cols] fp32 (or bf16 bits) -> (codes uint8 [rows, cols], e8m0 uint8 [rows, cols/32])."""
    x = _c(x, np.uint16 if is_bf16 else np.float32)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.uint8)
    e8 = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_combine_encode(x.ctypes.data, int(bool(is_bf16)), rows, cols, int(signs),
                             _p(codes, _u8p), _p(e8, _u8p))
    return codes, e8


def combine_decode(codes, e8m0, k, signs):
    """codes [tokens*k, cols], e8m0 [tokens*k, cols/32] -> fp32 [tokens, cols]: the k arrivals
    of each token summed, then rotated back."""
    codes = _c(codes, np.uint8)
    e8m0 = _c(e8m0, np.uint8)
    rows, cols = codes.shape
    assert rows % k == 0
    out = np.zeros((rows // k, cols), np.float32)
    lib().orc_combine_decode(_p(codes, _u8p), _p(e8m0, _u8p), rows // k, k, cols, int(signs), _p(out, _f32p))
    return out


# ---------------------------------------------------------------- MXFP4
def quantize_mxfp4(x, rht=False, signs=0):
    """bf16 bits [rows, cols] -> (codes [rows, cols/2], e8m0 [rows, cols/32]); rht rotates each
    group of 32 first."""
    x = _c(x, np.uint16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    e8 = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_quantize_mxfp4(_p(x, _u16p), rows, cols, cols, int(bool(rht)), int(signs), _p(codes, _u8p),
                             _p(e8, _u8p))
    return codes, e8


def dequant_mxfp4(codes, e8m0):
    codes = _c(codes, np.uint8)
    e8m0 = _c(e8m0, np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_mxfp4(_p(codes, _u8p), _p(e8m0, _u8p), rows, cols, _p(out, _f64p))
    return out


def gemm_mxfp4(a_codes, a_e8m0, b_codes, b_e8m0, with_abs=False):
    """D = A . B^T on exactly dequantized MXFP4 operands, float64."""
    return _product(dequant_mxfp4(a_codes, a_e8m0), dequant_mxfp4(b_codes, b_e8m0), with_abs)


# ---------------------------------------------------------------- GELU
def normal_cdf(x):
    return lib().orc_normal_cdf(float(x))


def normal_pdf(x):
    return lib().orc_normal_pdf(float(x))


def gelu(x):
    """GELU(x) = x Phi(x) (exact-erf form), float64."""
    return lib().orc_gelu(float(x))


def gelu_grad(x):
    """GELU'(x) = Phi(x) + x phi(x), float64."""
    return lib().orc_gelu_grad(float(x))


def gelu_bf16(h_bits, grad=False):
    """GELU (or GELU') of bf16 bit patterns, float64, same shape."""
    h = _c(h_bits, np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().orc_gelu_bf16(_p(h, _u16p), h.size, 1 if grad else 0, _p(out, _f64p))
    return out


# ---------------------------------------------------------------- GEMMs
# Each GEMM reference returns D = A . B^T on exactly dequantized operands (float64). With
# with_abs=True it returns (D, |A| . |B|^T, K): also the sum of |a_k b_k| behind every output
# element (the scale of the rounding error an fp32 accumulation of that element can carry)
# and the contraction length.
def _product(A, B, with_abs):
    D = A @ B.T
    return (D, np.abs(A) @ np.abs(B).T, A.shape[1]) if with_abs else D


def gemm_nvfp4(a_codes, a_scales, a_kind, a_sdec, b_codes, b_scales, b_kind, b_sdec, with_abs=False):
    """D = A . B^T on exactly dequantized NVFP4 operands, float64."""
    A = dequant_nvfp4(a_codes, a_scales, a_kind, a_sdec)
    B = dequant_nvfp4(b_codes, b_scales, b_kind, b_sdec)
    return _product(A, B, with_abs)


def gemm_nvfp4_rows(a_codes, a_scales, a_sdec_rows, b_codes, b_scales, b_kind, b_sdec, with_abs=False):
    """D = A . B^T with A carrying a per-row outer scale, float64."""
    A = dequant_nvfp4_rows(a_codes, a_scales, a_sdec_rows)
    B = dequant_nvfp4(b_codes, b_scales, b_kind, b_sdec)
    return _product(A, B, with_abs)


def gemm_mxfp8(a_e4m3, a_e8m0, b_e4m3, b_e8m0, with_abs=False):
    """D = A . B^T on exactly dequantized MXFP8 operands, float64."""
    return _product(dequant_mxfp8(a_e4m3, a_e8m0), dequant_mxfp8(b_e4m3, b_e8m0), with_abs)


def round_bf16(x):
    """float -> nearest-even bf16, returned as float32 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("ctypes", "os", "np", "lib")]
__all__ += ["lib"]
