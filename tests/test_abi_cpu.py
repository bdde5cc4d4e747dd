"""CPU checks of the C-ABI library: it loads, it exports every symbol include/fp4q.h
declares, and its host-side validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp4q.h")


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as g
    g.build()
    from mxfp8_precision_numerics_gb300 import fp4q
    return fp4q


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FP4Q_API\s+[\w\s\*]+?\b(fp4q_\w+)\s*\(", text)


def test_header_declares_the_six_entry_points():
    syms = set(declared_symbols())
    for name in ("fp4q_quantize_1d", "fp4q_quantize_2d", "fp4q_requant_t_mxfp8_sr", "fp4q_rht16",
                 "fp4q_gemm_nvfp4", "fp4q_gemm_mxfp8"):
        assert name in syms


def test_library_exports_every_declared_symbol(F):
    lib = ctypes.CDLL(F.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings_and_version(F):
    assert F.version() == 100
    for s in range(8):
        assert F.status_str(s).startswith("FP4Q")
    assert "unknown" in F.status_str(99)


def _lib(F):
    return F._lib


def test_requant_dual_validates_before_any_launch(F):
    L = _lib(F)
    p = ctypes.c_void_p(256)
    assert L.fp4q_requant_bf16_dual(None, 64, 64, 1, 0, 1, 0, 2, 3, p, p, p, p, None) == F.ERR_NULL
    assert L.fp4q_requant_bf16_dual(p, 64, 64, 2, 0, 1, 0, 2, 3, p, p, p, p, None) == F.ERR_ARG
    assert L.fp4q_requant_bf16_dual(p, 64, 64, 1, 0x10000, 1, 0, 2, 3, p, p, p, p, None) == F.ERR_ARG
    assert L.fp4q_requant_bf16_dual(p, 48, 64, 1, 0, 1, 0, 2, 3, p, p, p, p, None) == F.ERR_SHAPE
    assert L.fp4q_requant_bf16_dual(ctypes.c_void_p(264), 64, 64, 1, 0, 1, 0, 2, 3, p, p, p, p, None) == F.ERR_ALIGN


def test_wait_timeout_test_hook_validates_before_any_launch(F):
    L = _lib(F)
    p = ctypes.c_void_p(256)
    assert L.fp4q_test_gemm_wait_timeout(None, p, p, p, p, 512, 512, 1024, 20_000_000, None) == F.ERR_NULL
    assert L.fp4q_test_gemm_wait_timeout(p, p, p, p, p, 512, 512, 1024, 10, None) == F.ERR_ARG
    assert L.fp4q_test_gemm_wait_timeout(p, p, p, p, p, 512, 512, 1024, 3_000_000_000, None) == F.ERR_ARG
    assert L.fp4q_test_gemm_wait_timeout(p, p, p, p, p, 128, 512, 1024, 20_000_000, None) == F.ERR_SHAPE
    assert L.fp4q_test_gemm_wait_timeout(p, p, p, p, p, 512, 512, 640, 20_000_000, None) == F.ERR_SHAPE
    assert L.fp4q_test_gemm_wait_timeout(ctypes.c_void_p(264), p, p, p, p, 512, 512, 1024, 20_000_000,
                                         None) == F.ERR_ALIGN


def test_validation_rejects_bad_arguments_without_touching_cuda(F):
    L = _lib(F)
    p = ctypes.c_void_p(16)            # an aligned dummy address: never dereferenced
    q = ctypes.c_void_p(17)            # misaligned
    n = None
    # quantize_1d: NULL, shape, alignment
    assert L.fp4q_quantize_1d(n, 16, 32, 32, n, p, p, p, p, n) == F.ERR_NULL
    assert L.fp4q_quantize_1d(p, 16, 32, 32, n, n, p, p, p, n) == F.ERR_NULL   # no amax source
    assert L.fp4q_quantize_1d(p, 16, 40, 40, n, p, p, p, p, n) == F.ERR_SHAPE
    assert L.fp4q_quantize_1d(p, 0, 32, 32, n, p, p, p, p, n) == F.ERR_SHAPE
    assert L.fp4q_quantize_1d(p, 16, 32, 16, n, p, p, p, p, n) == F.ERR_SHAPE  # ld < cols
    assert L.fp4q_quantize_1d(q, 16, 32, 32, n, p, p, p, p, n) == F.ERR_ALIGN
    assert L.fp4q_quantize_1d(p, 16, 32, 36, n, p, p, p, p, n) == F.ERR_ALIGN  # ld % 8
    # quantize_2d
    assert L.fp4q_quantize_2d(p, 24, 32, 32, 1, 0, n, p, p, p, p, n) == F.ERR_SHAPE
    assert L.fp4q_quantize_2d(p, 32, 32, 32, 2, 16, n, p, p, p, p, n) == F.ERR_SHAPE  # overlapping batch
    assert L.fp4q_quantize_2d(p, 32, 32, 32, 1, 0, n, p, n, p, p, n) == F.ERR_NULL
    # requant
    assert L.fp4q_requant_t_mxfp8_sr(4, p, p, p, 32, 32, 1, 0, 0, 1, 0, 0, p, p, n) == F.ERR_ARG
    assert L.fp4q_requant_t_mxfp8_sr(3, p, p, n, 32, 32, 1, 0, 0, 1, 0, 0, p, p, n) == F.ERR_NULL  # s_dec rows
    assert L.fp4q_requant_t_mxfp8_sr(0, p, n, n, 32, 32, 2, 0, 0, 1, 0, 0, p, p, n) == F.ERR_ARG
    assert L.fp4q_requant_t_mxfp8_sr(0, p, n, n, 32, 32, 1, 0, 0, 2, 0, 0, p, p, n) == F.ERR_ARG
    assert L.fp4q_requant_t_mxfp8_sr(0, p, n, n, 32, 32, 1, 1, 1 << 16, 1, 0, 0, p, p, n) == F.ERR_ARG
    assert L.fp4q_requant_t_mxfp8_sr(1, p, n, p, 32, 32, 1, 0, 0, 1, 0, 0, p, p, n) == F.ERR_NULL
    assert L.fp4q_requant_t_mxfp8_sr(0, p, n, n, 48, 32, 1, 0, 0, 1, 0, 0, p, p, n) == F.ERR_SHAPE
    assert L.fp4q_requant_t_mxfp8_sr(0, p, n, n, 32, 32, 1, 0, 0, 1, 0, 0, q, p, n) == F.ERR_ALIGN
    # rht16
    assert L.fp4q_rht16(p, 2, p, 4, 16, 0, n) == F.ERR_ARG
    assert L.fp4q_rht16(p, 0, p, 4, 24, 0, n) == F.ERR_SHAPE
    assert L.fp4q_rht16(p, 0, q, 4, 16, 0, n) == F.ERR_ALIGN
    # gemm_nvfp4
    g = L.fp4q_gemm_nvfp4
    assert g(p, p, p, p, p, 3, p, p, 0, 128, 256, 256, 1, None, n) == F.ERR_ARG
    assert g(p, p, p, p, p, 1, p, p, 2, 128, 256, 256, 1, None, n) == F.ERR_ARG
    assert g(p, p, p, p, p, 1, p, p, 0, 128, 256, 128, 1, None, n) == F.ERR_SHAPE   # K % 256
    assert g(p, p, p, p, p, 1, p, p, 0, 128, 24, 256, 1, None, n) == F.ERR_SHAPE    # N % 16
    assert g(p, p, p, p, p, 1, p, p, 0, 128, 256, 256, 0, None, n) == F.ERR_ARG     # groups
    assert g(p, p, p, p, p, 1, p, p, 0, 128, 256, 256, 2, None, n) == F.ERR_NULL    # offsets
    offs = (ctypes.c_int64 * 3)(0, 100, 120)
    assert g(p, p, p, p, p, 1, p, p, 0, 128, 256, 256, 2, offs, n) == F.ERR_SHAPE   # last != M
    offs = (ctypes.c_int64 * 3)(0, 100, 64)
    assert g(p, p, p, p, p, 1, p, p, 0, 64, 256, 256, 2, offs, n) == F.ERR_SHAPE    # descending
    assert g(q, p, p, p, p, 1, p, p, 0, 128, 256, 256, 1, None, n) == F.ERR_ALIGN
    # gemm_mxfp8
    m = L.fp4q_gemm_mxfp8
    assert m(p, p, p, p, p, 0, 128, 256, 96, n) == F.ERR_SHAPE
    assert m(p, p, p, p, n, 0, 128, 256, 128, n) == F.ERR_NULL
    assert m(p, ctypes.c_void_p(18), p, p, p, 0, 128, 256, 128, n) == F.ERR_ALIGN
    # the fused-epilogue GEMMs
    ge = L.fp4q_gemm_nvfp4_gelu
    assert ge(p, p, p, p, p, 2, p, p, n, p, 128, 256, 256, n) == F.ERR_NULL           # no act_out
    assert ge(p, p, p, p, p, 2, p, p, p, n, 128, 256, 256, n) == F.ERR_NULL           # no amax
    assert ge(p, p, p, p, p, 3, p, p, p, p, 128, 256, 256, n) == F.ERR_ARG            # scale kind
    assert ge(p, p, p, p, p, 2, p, p, p, p, 128, 256, 200, n) == F.ERR_SHAPE          # K % 256
    assert ge(p, p, p, p, p, 2, p, p, q, p, 128, 256, 256, n) == F.ERR_ALIGN          # h_out
    gr = L.fp4q_gemm_nvfp4_gelu_rows
    assert gr(p, p, n, p, p, 2, p, p, p, n, 128, 256, 256, n) == F.ERR_NULL           # no row scales
    assert gr(p, p, p, p, p, 2, p, p, p, ctypes.c_void_p(18), 128, 256, 256, n) == F.ERR_ALIGN
    assert gr(p, p, p, p, p, 2, p, p, p, p, 128, 256, 200, n) == F.ERR_SHAPE          # K % 256
    # act_amax may be NULL in the per-row form: past validation, no GPU here
    assert gr(p, p, p, p, p, 2, p, p, p, n, 128, 256, 256, n) in (F.ERR_CUDA, F.ERR_UNSUPPORTED)
    r = L.fp4q_gemm_nvfp4_rows
    assert r(p, p, n, p, p, 1, p, p, 0, 128, 256, 256, 1, None, n) == F.ERR_NULL
    assert r(p, p, p, p, p, 3, p, p, 0, 128, 256, 256, 1, None, n) == F.ERR_ARG
    assert r(p, p, p, p, p, 1, p, p, 0, 128, 256, 128, 1, None, n) == F.ERR_SHAPE
    # quantize_1d_rows
    qr = L.fp4q_quantize_1d_rows
    assert qr(p, 16, 32, 32, 2, p, p, p, n) == F.ERR_ARG                               # four_six
    assert qr(p, 16, 32, 32, 1, p, p, n, n) == F.ERR_NULL
    assert qr(p, 16, 40, 40, 1, p, p, p, n) == F.ERR_SHAPE
    assert qr(p, 0, 32, 32, 1, p, p, p, n) == F.ERR_SHAPE
    assert qr(p, 16, 32, 16, 1, p, p, p, n) == F.ERR_SHAPE                             # ld < cols
    assert qr(q, 16, 32, 32, 1, p, p, p, n) == F.ERR_ALIGN
    assert qr(p, 16, 32, 36, 1, p, p, p, n) == F.ERR_ALIGN                             # ld % 8
    assert qr(p, 16, 32, 32, 1, p, p, p, n) in (F.ERR_CUDA, F.ERR_UNSUPPORTED)        # valid, no GPU
    # MXFP4
    qm = L.fp4q_quantize_mxfp4
    assert qm(p, 4, 64, 64, 2, 0, p, p, n) == F.ERR_ARG
    assert qm(p, 4, 48, 48, 0, 0, p, p, n) == F.ERR_SHAPE
    assert qm(p, 4, 64, 64, 0, 0, p, n, n) == F.ERR_NULL
    assert qm(p, 4, 64, 68, 0, 0, p, p, n) == F.ERR_ALIGN
    gm = L.fp4q_gemm_mxfp4
    assert gm(p, p, p, p, p, 0, 128, 256, 1024, n) == F.ERR_SHAPE                    # K % 2048
    assert gm(p, p, p, p, p, 0, 128, 24, 2048, n) == F.ERR_SHAPE
    assert gm(p, p, p, p, p, 2, 128, 256, 2048, n) == F.ERR_ARG
    assert gm(p, n, p, p, p, 0, 128, 256, 2048, n) == F.ERR_NULL
    assert gm(p, ctypes.c_void_p(20), p, p, p, 0, 128, 256, 2048, n) == F.ERR_ALIGN
    # combine codec
    ce = L.fp4q_combine_encode
    assert ce(p, 2, 4, 64, 0, p, p, n) == F.ERR_ARG                                    # dtype
    assert ce(p, 0, 4, 48, 0, p, p, n) == F.ERR_SHAPE                                  # cols % 32
    assert ce(p, 0, 0, 64, 0, p, p, n) == F.ERR_SHAPE
    assert ce(p, 0, 4, 64, 0, n, p, n) == F.ERR_NULL
    assert ce(q, 0, 4, 64, 0, p, p, n) == F.ERR_ALIGN
    cd = L.fp4q_combine_decode
    assert cd(p, p, 4, 0, 64, 0, p, 0, n) == F.ERR_SHAPE                               # k
    assert cd(p, p, 4, 2, 40, 0, p, 0, n) == F.ERR_SHAPE
    assert cd(p, p, 4, 2, 64, 0, p, 3, n) == F.ERR_ARG
    assert cd(p, n, 4, 2, 64, 0, p, 0, n) == F.ERR_NULL
    assert cd(p, p, 4, 2, 64, 0, q, 0, n) == F.ERR_ALIGN
    gc = L.fp4q_gemm_nvfp4_combine
    assert gc(p, p, p, p, p, 2, p, 0, p, p, 128, 48, 256, 1, None, n) == F.ERR_SHAPE  # N % 32
    assert gc(p, p, p, p, p, 2, p, 0, p, n, 128, 64, 256, 1, None, n) == F.ERR_NULL
    assert gc(p, p, p, p, p, 3, p, 0, p, p, 128, 64, 256, 1, None, n) == F.ERR_ARG
    assert gc(p, p, p, p, p, 2, p, 0, q, p, 128, 64, 256, 1, None, n) == F.ERR_ALIGN
    dg = L.fp4q_gemm_mxfp8_dgelu
    assert dg(p, p, p, p, n, p, 128, 256, 128, n) == F.ERR_NULL                        # no h
    assert dg(p, p, p, p, p, p, 128, 250, 128, n) == F.ERR_SHAPE                       # N % 16
    assert dg(p, p, p, p, p, q, 128, 256, 128, n) == F.ERR_ALIGN                       # dh_out


def test_product_path_has_no_oracle_or_fallback():
    """The CUDA library and its binding never reach the oracle or a CPU path."""
    pkg = os.path.join(ROOT, "mxfp8_precision_numerics_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f


def test_empty_inputs_are_rejected_before_any_launch(F):
    """A zero (or negative) size in any dimension is FP4Q_ERR_SHAPE at every entry point, checked
    on the host: no kernel is launched for an empty tensor (the header states the minimum sizes)."""
    L = _lib(F)
    p = ctypes.c_void_p(256)
    n = None
    S = F.ERR_SHAPE
    for rows, cols in ((0, 32), (16, 0), (-16, 32)):
        assert L.fp4q_quantize_1d(p, rows, cols, 32, n, p, p, p, p, n) == S
        assert L.fp4q_quantize_1d_rows(p, rows, cols, 32, 1, p, p, p, n) == S
        assert L.fp4q_quantize_2d(p, rows, cols, 32, 1, 0, n, p, p, p, p, n) == S
        assert L.fp4q_quantize_2d_noalloc(p, rows, cols, 32, 1, 0, p, p, p, n) == S
        assert L.fp4q_quantize_mxfp4(p, rows, cols, 32, 0, 0, p, p, n) == S
        assert L.fp4q_rht16(p, 0, p, rows, cols, 0, n) == S
        assert L.fp4q_combine_encode(p, 0, rows, cols, 0, p, p, n) == S
    for rows, cols in ((0, 64), (64, 0)):
        for kind in (0, 1, 2):
            assert L.fp4q_requant_t_mxfp8_sr(kind, p, p, p, rows, cols, 1, 0, 0, 1, 0, 0, p, p, n) == S
        assert L.fp4q_requant_bf16_dual(p, rows, cols, 1, 0, 1, 0, 2, 3, p, p, p, p, n) == S
    assert L.fp4q_combine_decode(p, p, 0, 2, 64, 0, p, 0, n) == S
    for M, N, K in ((0, 256, 256), (128, 0, 256), (128, 256, 0)):
        assert L.fp4q_gemm_nvfp4(p, p, p, p, p, 1, p, p, 0, M, N, K, 1, None, n) == S
        assert L.fp4q_gemm_nvfp4_rows(p, p, p, p, p, 1, p, p, 0, M, N, K, 1, None, n) == S
        assert L.fp4q_gemm_nvfp4_gelu(p, p, p, p, p, 2, p, p, p, p, M, N, K, n) == S
        assert L.fp4q_gemm_mxfp8(p, p, p, p, p, 0, M, N, K, n) == S
        assert L.fp4q_gemm_mxfp8_dgelu(p, p, p, p, p, p, M, N, K, n) == S
        assert L.fp4q_gemm_mxfp4(p, p, p, p, p, 0, M, N, max(K, 0) * 8, n) == S
