"""ctypes binding over ``libfp4q.so`` (the C ABI of ``include/fp4q.h``).

Argument marshalling only: every function passes device pointers, sizes and the
current CUDA stream straight to the library, and every step of the computation runs
in the library's kernels. Importing this module loads the library and raises if it
has not been built: there is no fallback path.

Low-level functions carry the ABI names (``fp4q_quantize_1d`` ...) and take
caller-allocated torch tensors for every buffer. The convenience functions without
the prefix allocate their outputs with torch (device memory is plumbing) and return
them.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp4q.so")

OK, ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_ARG, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(8)
IN_BF16, IN_NVFP4_1D, IN_NVFP4_2D, IN_NVFP4_1D_ROWS = 0, 1, 2, 3
RNE, SR = 0, 1
F32, BF16 = 0, 1
SCALE_1D, SCALE_2D = 1, 2
NOALLOC_MAX_BATCH = 1024      # FP4Q_NOALLOC_MAX_BATCH

# tensor tags of the four backward quantizations (stochastic-rounding counter streams)
TAG_WT, TAG_DY_ROWS, TAG_DY_T, TAG_XT = 1, 2, 3, 4

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "(the CUDA library is required; there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64

_SIGS = {
    "fp4q_status_str": (ctypes.c_char_p, [_int]),
    "fp4q_version": (_int, []),
    "fp4q_quantize_1d": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fp4q_quantize_1d_rows": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _vp, _vp, _vp]),
    "fp4q_quantize_2d": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fp4q_quantize_2d_noalloc": (_int, [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fp4q_requant_t_mxfp8_sr": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _int, _int, _u32, _int, _u64,
                                       _u32, _vp, _vp, _vp]),
    "fp4q_rht16": (_int, [_vp, _int, _vp, _i64, _i64, _u32, _vp]),
    "fp4q_requant_bf16_dual": (_int, [_vp, _i64, _i64, _int, _u32, _int, _u64, _u32, _u32, _vp, _vp, _vp, _vp, _vp]),
    "fp4q_gemm_nvfp4": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _i64, _i64, _int,
                               ctypes.POINTER(ctypes.c_int64), _vp]),
    "fp4q_gemm_nvfp4_rows": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _i64, _i64, _int,
                                    _vp, _vp]),
    "fp4q_gemm_mxfp8": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp]),
    "fp4q_gemm_nvfp4_gelu": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "fp4q_gemm_nvfp4_gelu_rows": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                         _vp]),
    "fp4q_gemm_mxfp8_dgelu": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "fp4q_quantize_mxfp4": (_int, [_vp, _i64, _i64, _i64, _int, _u32, _vp, _vp, _vp]),
    "fp4q_gemm_mxfp4": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp]),
    "fp4q_combine_encode": (_int, [_vp, _int, _i64, _i64, _u32, _vp, _vp, _vp]),
    "fp4q_combine_decode": (_int, [_vp, _vp, _i64, _i64, _i64, _u32, _vp, _int, _vp]),
    "fp4q_gemm_nvfp4_combine": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _u32, _vp, _vp, _i64, _i64, _i64,
                                       _int, _vp, _vp]),
    "fp4q_device_status": (_int, [_vp]),
    "fp4q_test_gemm_wait_timeout": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class Fp4qError(RuntimeError):
    def __init__(self, status, where):
        super().__init__(f"{where}: {status_str(status)}")
        self.status = status


def status_str(status):
    return _lib.fp4q_status_str(int(status)).decode()


def version():
    return _lib.fp4q_version()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != OK:
        raise Fp4qError(status, where)


# ------------------------------------------------------------------ raw ABI calls
def fp4q_quantize_1d(x, rows, cols, ld, amax_in, amax_ws, codes, scales, s_dec_out, stream=None):
    _check(_lib.fp4q_quantize_1d(_ptr(x), rows, cols, ld, _ptr(amax_in), _ptr(amax_ws), _ptr(codes),
                                 _ptr(scales), _ptr(s_dec_out), _stream(stream)), "fp4q_quantize_1d")


def fp4q_quantize_1d_rows(x, rows, cols, ld, four_six, codes, scales, s_dec_rows, stream=None):
    _check(_lib.fp4q_quantize_1d_rows(_ptr(x), rows, cols, ld, int(four_six), _ptr(codes), _ptr(scales),
                                      _ptr(s_dec_rows), _stream(stream)), "fp4q_quantize_1d_rows")


def fp4q_quantize_2d(w, rows, cols, ld, batch, batch_stride, amax_in, amax_ws, codes, tile_scales,
                     s_dec_out, stream=None):
    _check(_lib.fp4q_quantize_2d(_ptr(w), rows, cols, ld, batch, batch_stride, _ptr(amax_in),
                                 _ptr(amax_ws), _ptr(codes), _ptr(tile_scales), _ptr(s_dec_out),
                                 _stream(stream)), "fp4q_quantize_2d")


def fp4q_quantize_2d_noalloc(w, rows, cols, ld, batch, batch_stride, codes, tile_scales, s_dec_out,
                             stream=None):
    """fp4q_quantize_2d with the amax workspace inside the library (for callers that cannot
    allocate device memory); batch <= NOALLOC_MAX_BATCH."""
    _check(_lib.fp4q_quantize_2d_noalloc(_ptr(w), rows, cols, ld, batch, batch_stride, _ptr(codes),
                                         _ptr(tile_scales), _ptr(s_dec_out), _stream(stream)),
           "fp4q_quantize_2d_noalloc")


def fp4q_requant_t_mxfp8_sr(in_kind, inp, in_scales, in_s_dec, rows, cols, transpose, rht, rht_signs,
                            rounding, seed, tag, out_e4m3, out_e8m0, stream=None):
    _check(_lib.fp4q_requant_t_mxfp8_sr(in_kind, _ptr(inp), _ptr(in_scales), _ptr(in_s_dec), rows, cols,
                                        int(transpose), int(rht), int(rht_signs), rounding,
                                        int(seed) & ((1 << 64) - 1), int(tag), _ptr(out_e4m3),
                                        _ptr(out_e8m0), _stream(stream)), "fp4q_requant_t_mxfp8_sr")


def fp4q_rht16(inp, in_dtype, out, rows, cols, signs, stream=None):
    _check(_lib.fp4q_rht16(_ptr(inp), in_dtype, _ptr(out), rows, cols, int(signs), _stream(stream)),
           "fp4q_rht16")


def fp4q_requant_bf16_dual(inp, rows, cols, rht, rht_signs, rounding, seed, tag_rows, tag_t, rows_e4m3, rows_e8m0,
                           t_e4m3, t_e8m0, stream=None):
    _check(_lib.fp4q_requant_bf16_dual(_ptr(inp), rows, cols, int(rht), int(rht_signs), rounding, int(seed),
                                       int(tag_rows), int(tag_t), _ptr(rows_e4m3), _ptr(rows_e8m0), _ptr(t_e4m3),
                                       _ptr(t_e8m0), _stream(stream)), "fp4q_requant_bf16_dual")


def _offsets(group_row_offsets):
    if group_row_offsets is None:
        return None, None
    arr = (ctypes.c_int64 * len(group_row_offsets))(*[int(v) for v in group_row_offsets])
    return arr, ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64))


def fp4q_gemm_nvfp4(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, d, d_dtype, M, N, K,
                    groups=1, group_row_offsets=None, stream=None):
    keep, offs = _offsets(group_row_offsets)
    _check(_lib.fp4q_gemm_nvfp4(_ptr(a), _ptr(a_scales), _ptr(a_s_dec), _ptr(b), _ptr(b_scales),
                                b_scale_kind, _ptr(b_s_dec), _ptr(d), d_dtype, M, N, K, groups, offs,
                                _stream(stream)), "fp4q_gemm_nvfp4")
    del keep


def fp4q_gemm_nvfp4_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, d, d_dtype, M, N, K,
                         groups=1, group_row_offsets=None, stream=None):
    keep, offs = _offsets(group_row_offsets)
    _check(_lib.fp4q_gemm_nvfp4_rows(_ptr(a), _ptr(a_scales), _ptr(a_s_dec_rows), _ptr(b), _ptr(b_scales),
                                     b_scale_kind, _ptr(b_s_dec), _ptr(d), d_dtype, M, N, K, groups, offs,
                                     _stream(stream)), "fp4q_gemm_nvfp4_rows")
    del keep


def fp4q_gemm_mxfp8(a, a_scales, b, b_scales, d, d_dtype, M, N, K, stream=None):
    _check(_lib.fp4q_gemm_mxfp8(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), _ptr(d), d_dtype,
                                M, N, K, _stream(stream)), "fp4q_gemm_mxfp8")


def fp4q_gemm_nvfp4_gelu(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, h_out, act_out, act_amax,
                         M, N, K, stream=None):
    _check(_lib.fp4q_gemm_nvfp4_gelu(_ptr(a), _ptr(a_scales), _ptr(a_s_dec), _ptr(b), _ptr(b_scales),
                                     b_scale_kind, _ptr(b_s_dec), _ptr(h_out), _ptr(act_out), _ptr(act_amax),
                                     M, N, K, _stream(stream)), "fp4q_gemm_nvfp4_gelu")


def fp4q_gemm_nvfp4_gelu_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, h_out, act_out,
                              act_amax, M, N, K, stream=None):
    _check(_lib.fp4q_gemm_nvfp4_gelu_rows(_ptr(a), _ptr(a_scales), _ptr(a_s_dec_rows), _ptr(b), _ptr(b_scales),
                                          b_scale_kind, _ptr(b_s_dec), _ptr(h_out), _ptr(act_out),
                                          _ptr(act_amax), M, N, K, _stream(stream)),
           "fp4q_gemm_nvfp4_gelu_rows")


def fp4q_gemm_mxfp8_dgelu(a, a_scales, b, b_scales, h, dh_out, M, N, K, stream=None):
    _check(_lib.fp4q_gemm_mxfp8_dgelu(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), _ptr(h), _ptr(dh_out),
                                      M, N, K, _stream(stream)), "fp4q_gemm_mxfp8_dgelu")


def fp4q_quantize_mxfp4(x, rows, cols, ld, rht, rht_signs, codes, e8m0, stream=None):
    _check(_lib.fp4q_quantize_mxfp4(_ptr(x), rows, cols, ld, int(rht), int(rht_signs), _ptr(codes), _ptr(e8m0),
                                    _stream(stream)), "fp4q_quantize_mxfp4")


def fp4q_gemm_mxfp4(a, a_e8m0, b, b_e8m0, d, d_dtype, M, N, K, stream=None):
    _check(_lib.fp4q_gemm_mxfp4(_ptr(a), _ptr(a_e8m0), _ptr(b), _ptr(b_e8m0), _ptr(d), d_dtype, M, N, K,
                                _stream(stream)), "fp4q_gemm_mxfp4")


def fp4q_combine_encode(x, x_dtype, rows, cols, rht_signs, codes, e8m0, stream=None):
    _check(_lib.fp4q_combine_encode(_ptr(x), x_dtype, rows, cols, int(rht_signs), _ptr(codes), _ptr(e8m0),
                                    _stream(stream)), "fp4q_combine_encode")


def fp4q_combine_decode(codes, e8m0, tokens, k, cols, rht_signs, out, out_dtype, stream=None):
    _check(_lib.fp4q_combine_decode(_ptr(codes), _ptr(e8m0), tokens, k, cols, int(rht_signs), _ptr(out),
                                    out_dtype, _stream(stream)), "fp4q_combine_decode")


def fp4q_gemm_nvfp4_combine(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, rht_signs, codes_out,
                            e8m0_out, M, N, K, groups=1, group_row_offsets=None, stream=None):
    keep, offs = _offsets(group_row_offsets)
    _check(_lib.fp4q_gemm_nvfp4_combine(_ptr(a), _ptr(a_scales), _ptr(a_s_dec), _ptr(b), _ptr(b_scales),
                                        b_scale_kind, _ptr(b_s_dec), int(rht_signs), _ptr(codes_out),
                                        _ptr(e8m0_out), M, N, K, groups, offs, _stream(stream)),
           "fp4q_gemm_nvfp4_combine")
    del keep


def fp4q_device_status(stream=None):
    return _lib.fp4q_device_status(_stream(stream))


def fp4q_test_gemm_wait_timeout(a, a_scales, b, b_scales, d, M, N, K, wait_limit_ns, stream=None):
    """The failure-detection test launch (returns the launch status; fp4q_device_status then
    reports FP4Q_ERR_TIMEOUT)."""
    return _lib.fp4q_test_gemm_wait_timeout(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), _ptr(d), M, N, K,
                                            int(wait_limit_ns), _stream(stream))


# ------------------------------------------------------------------ allocating helpers
def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def quantize_1d(x, amax_in=None, stream=None):
    """bf16 [rows, cols] -> (codes u8 [rows, cols/2], scales u8 [rows, cols/16], s_dec f32 [1],
    amax f32 [1])."""
    rows, cols = x.shape
    dev = x.device
    codes = _empty((rows, cols // 2), torch.uint8, dev)
    scales = _empty((rows, cols // 16), torch.uint8, dev)
    s_dec = _empty((1,), torch.float32, dev)
    amax_ws = None if amax_in is not None else _empty((1,), torch.float32, dev)
    fp4q_quantize_1d(x, rows, cols, x.stride(0), amax_in, amax_ws, codes, scales, s_dec, stream)
    return codes, scales, s_dec, (amax_in if amax_in is not None else amax_ws)


def quantize_1d_rows(x, four_six=True, stream=None):
    """bf16 [rows, cols] -> (codes u8 [rows, cols/2], scales u8 [rows, cols/16],
    s_dec_rows f32 [rows]): one outer scale per row, 4/6 block scales if four_six."""
    rows, cols = x.shape
    dev = x.device
    codes = _empty((rows, cols // 2), torch.uint8, dev)
    scales = _empty((rows, cols // 16), torch.uint8, dev)
    s_dec = _empty((rows,), torch.float32, dev)
    fp4q_quantize_1d_rows(x, rows, cols, x.stride(0), four_six, codes, scales, s_dec, stream)
    return codes, scales, s_dec


def quantize_2d(w, amax_in=None, stream=None):
    """bf16 [rows, cols] or [batch, rows, cols] -> (codes, tile_scales, s_dec [batch], amax)."""
    batched = w.dim() == 3
    w3 = w if batched else w.unsqueeze(0)
    batch, rows, cols = w3.shape
    dev = w.device
    codes = _empty((batch, rows, cols // 2), torch.uint8, dev)
    tiles = _empty((batch, rows // 16, cols // 16), torch.uint8, dev)
    s_dec = _empty((batch,), torch.float32, dev)
    amax_ws = None if amax_in is not None else _empty((batch,), torch.float32, dev)
    fp4q_quantize_2d(w3, rows, cols, w3.stride(1), batch, w3.stride(0), amax_in, amax_ws, codes, tiles,
                     s_dec, stream)
    if not batched:
        codes, tiles = codes[0], tiles[0]
    return codes, tiles, s_dec, (amax_in if amax_in is not None else amax_ws)


def requant_mxfp8(in_kind, inp, in_scales, in_s_dec, rows, cols, transpose, rht, rht_signs,
                  rounding, seed, tag, stream=None):
    """-> (e4m3 u8 [out_rows, out_cols], e8m0 u8 [out_rows, out_cols/32])."""
    orows, ocols = (cols, rows) if transpose else (rows, cols)
    dev = inp.device
    e4 = _empty((orows, ocols), torch.uint8, dev)
    e8 = _empty((orows, ocols // 32), torch.uint8, dev)
    fp4q_requant_t_mxfp8_sr(in_kind, inp, in_scales, in_s_dec, rows, cols, transpose, rht, rht_signs,
                            rounding, seed, tag, e4, e8, stream)
    return e4, e8


def requant_bf16_dual(inp, rht, rht_signs, rounding, seed, tag_rows, tag_t, stream=None):
    """bf16 [rows, cols] -> ((e4m3 [rows, cols], e8m0 [rows, cols/32]),
    (e4m3 [cols, rows], e8m0 [cols, rows/32])): the rowwise and the transposed requantization
    from one read."""
    rows, cols = inp.shape
    dev = inp.device
    r4 = _empty((rows, cols), torch.uint8, dev)
    r8 = _empty((rows, cols // 32), torch.uint8, dev)
    t4 = _empty((cols, rows), torch.uint8, dev)
    t8 = _empty((cols, rows // 32), torch.uint8, dev)
    fp4q_requant_bf16_dual(inp, rows, cols, rht, rht_signs, rounding, seed, tag_rows, tag_t, r4, r8, t4, t8, stream)
    return (r4, r8), (t4, t8)


def rht16(inp, signs, stream=None):
    rows, cols = inp.shape
    out = _empty((rows, cols), torch.float32, inp.device)
    fp4q_rht16(inp, BF16 if inp.dtype == torch.bfloat16 else F32, out, rows, cols, signs, stream)
    return out


def gemm_nvfp4(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, out_dtype=torch.float32,
               groups=1, group_row_offsets=None, stream=None):
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[-2]
    d = _empty((M, N), out_dtype, a.device)
    fp4q_gemm_nvfp4(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, d,
                    BF16 if out_dtype == torch.bfloat16 else F32, M, N, K, groups, group_row_offsets,
                    stream)
    return d


def gemm_nvfp4_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, out_dtype=torch.float32,
                    groups=1, group_row_offsets=None, stream=None):
    """gemm_nvfp4 with one outer scale per row of A (a_s_dec_rows f32 [M])."""
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[-2]
    d = _empty((M, N), out_dtype, a.device)
    fp4q_gemm_nvfp4_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, d,
                         BF16 if out_dtype == torch.bfloat16 else F32, M, N, K, groups, group_row_offsets,
                         stream)
    return d


def gemm_nvfp4_gelu_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, stream=None):
    """-> (h, act): gemm_nvfp4_gelu with one outer scale per row of A, no tensor amax."""
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[-2]
    h = _empty((M, N), torch.bfloat16, a.device)
    act = _empty((M, N), torch.bfloat16, a.device)
    fp4q_gemm_nvfp4_gelu_rows(a, a_scales, a_s_dec_rows, b, b_scales, b_scale_kind, b_s_dec, h, act, None,
                              M, N, K, stream)
    return h, act


def gemm_nvfp4_gelu(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, stream=None):
    """-> (h, act, act_amax): h = A.B^T in bf16, act = GELU(h) in bf16, act_amax = max|act|."""
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[-2]
    h = _empty((M, N), torch.bfloat16, a.device)
    act = _empty((M, N), torch.bfloat16, a.device)
    amax = _empty((1,), torch.float32, a.device)
    fp4q_gemm_nvfp4_gelu(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, h, act, amax, M, N, K, stream)
    return h, act, amax


def gemm_mxfp8_dgelu(a, a_scales, b, b_scales, h, stream=None):
    """-> dh = bf16(bf16(A.B^T) * GELU'(h)), bf16 [M][N]."""
    M, K = a.shape
    N = b.shape[0]
    dh = _empty((M, N), torch.bfloat16, a.device)
    fp4q_gemm_mxfp8_dgelu(a, a_scales, b, b_scales, h, dh, M, N, K, stream)
    return dh


def quantize_mxfp4(x, rht=False, rht_signs=0, stream=None):
    """bf16 [rows, cols] -> (codes u8 [rows, cols/2], e8m0 u8 [rows, cols/32])."""
    rows, cols = x.shape
    codes = _empty((rows, cols // 2), torch.uint8, x.device)
    e8 = _empty((rows, cols // 32), torch.uint8, x.device)
    fp4q_quantize_mxfp4(x, rows, cols, x.stride(0), rht, rht_signs, codes, e8, stream)
    return codes, e8


def gemm_mxfp4(a, a_e8m0, b, b_e8m0, out_dtype=torch.float32, stream=None):
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[0]
    d = _empty((M, N), out_dtype, a.device)
    fp4q_gemm_mxfp4(a, a_e8m0, b, b_e8m0, d, BF16 if out_dtype == torch.bfloat16 else F32, M, N, K, stream)
    return d


def combine_encode(x, rht_signs, stream=None):
    """fp32 or bf16 [rows, cols] -> (S2F6 codes u8 [rows, cols], e8m0 u8 [rows, cols/32])."""
    rows, cols = x.shape
    codes = _empty((rows, cols), torch.uint8, x.device)
    e8 = _empty((rows, cols // 32), torch.uint8, x.device)
    fp4q_combine_encode(x, BF16 if x.dtype == torch.bfloat16 else F32, rows, cols, rht_signs, codes, e8, stream)
    return codes, e8


def combine_decode(codes, e8m0, k, rht_signs, out_dtype=torch.float32, stream=None):
    """[tokens*k, cols] arrivals -> [tokens, cols]: each token's k arrivals summed, rotated back."""
    rows, cols = codes.shape
    out = _empty((rows // k, cols), out_dtype, codes.device)
    fp4q_combine_decode(codes, e8m0, rows // k, k, cols, rht_signs, out,
                        BF16 if out_dtype == torch.bfloat16 else F32, stream)
    return out


def gemm_nvfp4_combine(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, rht_signs, groups=1,
                       group_row_offsets=None, stream=None):
    """gemm_nvfp4 whose output leaves in the combine wire format -> (codes [M, N], e8m0 [M, N/32])."""
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[-2]
    codes = _empty((M, N), torch.uint8, a.device)
    e8 = _empty((M, N // 32), torch.uint8, a.device)
    fp4q_gemm_nvfp4_combine(a, a_scales, a_s_dec, b, b_scales, b_scale_kind, b_s_dec, rht_signs, codes, e8,
                            M, N, K, groups, group_row_offsets, stream)
    return codes, e8


def gemm_mxfp8(a, a_scales, b, b_scales, out_dtype=torch.float32, stream=None):
    M, K = a.shape
    N = b.shape[0]
    d = _empty((M, N), out_dtype, a.device)
    fp4q_gemm_mxfp8(a, a_scales, b, b_scales, d, BF16 if out_dtype == torch.bfloat16 else F32, M, N, K,
                    stream)
    return d
