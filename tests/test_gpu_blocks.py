"""Device building blocks against the oracle, element by element: the E2M1 and E4M3
encoders (every tie, saturation, the subnormal range), E4M3 stochastic rounding, the
MXFP8 ceiling exponent, and the Philox4x32-10 generator (also against cuRAND's own
implementation of the same published generator)."""
import ctypes

import numpy as np
import pytest
import torch

from helpers import assert_bytes_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import __graft_entry__ as g
    g.build()
    return ctypes.CDLL(g.PROBE_LIB)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def e2m1_inputs():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    vals = list(np.linspace(-8, 8, 40001, dtype=np.float32))
    for i in range(7):
        m = np.float32((grid[i] + grid[i + 1]) / 2)
        for v in (m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(9))):
            vals += [v, -v]
    vals += [0.0, -0.0, 6.0, 6.5, 1e30, -1e30, 1e-40, -1e-40, 5.0, 4.999999, 5.000001]
    return np.array(vals, dtype=np.float32)


def e4m3_inputs(rng):
    import oracle
    grid = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = [mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
            grid.astype(np.float32), np.array([448.0, 449.0, 463.99, 464.0, 465.0, 1e9, 0.0, -0.0],
                                              np.float32)]
    # random fp32 bit patterns spread over [2^-20, 2^9]
    e = rng.integers(107, 136, 200000)
    m = rng.integers(0, 1 << 23, 200000)
    vals.append(((e << 23) | m).astype(np.uint32).view(np.float32))
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v])


def test_e2m1_encoder_matches_oracle(P, orc):
    x = e2m1_inputs()
    n = len(x)
    xd = torch.from_numpy(x).cuda()
    alu = torch.empty(n, dtype=torch.uint8, device="cuda")
    lo = torch.empty_like(alu)
    hi = torch.empty_like(alu)
    assert P.probe_e2m1(_p(xd), _p(alu), _p(lo), _p(hi), n, _stream()) == 0
    torch.cuda.synchronize()
    want = np.array([orc.e2m1_encode_rne(v) for v in x], dtype=np.uint8)
    assert_bytes_equal(alu.cpu().numpy(), want, "E2M1 encoder (ALU)")
    # the hardware conversion the quantizers use: same codes, including every tie (the pages
    # report a hardware that breaks ties toward zero; on this device it must be to even),
    # with the first source operand in the high nibble
    lo, hi = lo.cpu().numpy(), hi.cpu().numpy()
    assert_bytes_equal(lo & 15, want, "E2M1 hardware cvt (low nibble)")
    assert_bytes_equal(lo >> 4, np.zeros_like(want), "E2M1 hardware cvt (other nibble)")
    assert_bytes_equal(hi >> 4, want, "E2M1 hardware cvt (high nibble)")


def test_e4m3_encoder_matches_oracle(P, orc):
    x = e4m3_inputs(np.random.default_rng(0))
    n = len(x)
    xd = torch.from_numpy(x).cuda()
    alu = torch.empty(n, dtype=torch.uint8, device="cuda")
    h1 = torch.empty(n, dtype=torch.int16, device="cuda")
    h2 = torch.empty_like(h1)
    assert P.probe_e4m3(_p(xd), _p(alu), _p(h1), _p(h2), n, _stream()) == 0
    torch.cuda.synchronize()
    lib = orc.lib()
    want = np.fromiter((lib.orc_e4m3_encode_rne_sat(float(v)) for v in x), dtype=np.uint8, count=n)
    assert_bytes_equal(alu.cpu().numpy(), want, "E4M3 encoder (ALU)")
    # the hardware E4M3 conversion agrees too (first operand -> high byte)
    h1 = h1.cpu().numpy().view(np.uint16)
    h2 = h2.cpu().numpy().view(np.uint16)
    assert_bytes_equal((h1 >> 8).astype(np.uint8), want, "E4M3 hardware cvt (high byte)")
    assert_bytes_equal((h2 & 0xFF).astype(np.uint8), want, "E4M3 hardware cvt (low byte)")


def test_e4m3_stochastic_rounding_matches_oracle(P, orc):
    rng = np.random.default_rng(1)
    x = e4m3_inputs(rng)
    x = x[np.abs(x) <= 448.0]
    n = len(x)
    r = rng.integers(0, 1 << 16, n).astype(np.uint32)
    r[:64] = [0, 1, 2, 65535, 65534, 32768, 32767, 4096] * 8
    xd = torch.from_numpy(x).cuda()
    rd = torch.from_numpy(r.view(np.int32)).cuda()
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert P.probe_e4m3_sr(_p(xd), _p(rd), _p(out), n, _stream()) == 0
    torch.cuda.synchronize()
    lib = orc.lib()
    want = np.fromiter((lib.orc_e4m3_encode_sr(float(v), int(k)) for v, k in zip(x, r)),
                       dtype=np.uint8, count=n)
    assert_bytes_equal(out.cpu().numpy(), want, "E4M3 stochastic rounding")


def test_mx_exponent_matches_oracle(P, orc):
    rng = np.random.default_rng(2)
    vals = [0.0, 1e-45, 1e-40, 2.0 ** -126, 448.0, 224.0, 448.0 * 2 ** -127, 3.4e38]
    for k in range(-140, 128, 3):
        edge = np.float32(448.0 * 2.0 ** k) if -149 < k + 8 < 128 else None
        if edge is not None and np.isfinite(edge) and edge > 0:
            vals += [edge, np.nextafter(edge, np.float32(np.inf)), np.nextafter(edge, np.float32(0))]
    e = rng.integers(1, 255, 100000)
    m = rng.integers(0, 1 << 23, 100000)
    vals = np.concatenate([np.array(vals, np.float32), ((e << 23) | m).astype(np.uint32).view(np.float32)])
    n = len(vals)
    vd = torch.from_numpy(vals).cuda()
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    assert P.probe_mx_exponent(_p(vd), _p(out), n, _stream()) == 0
    torch.cuda.synchronize()
    want = np.array([orc.pow2_ceil_exponent(float(v), 448.0) for v in vals], dtype=np.int32)
    got = out.cpu().numpy()
    bad = np.nonzero(got != want)[0]
    assert len(bad) == 0, f"{len(bad)} exponents differ, e.g. amax={vals[bad[0]]!r}: {got[bad[0]]} vs {want[bad[0]]}"


def test_philox_matches_oracle_and_curand(P, orc):
    rng = np.random.default_rng(3)
    n = 4096
    ctr = rng.integers(0, 1 << 32, (n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    key[0] = 0
    cd = torch.from_numpy(ctr.view(np.int32)).cuda()
    kd = torch.from_numpy(key.view(np.int32)).cuda()
    mine = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    ref = torch.empty_like(mine)
    assert P.probe_philox(_p(cd), _p(kd), _p(mine), _p(ref), n, _stream()) == 0
    torch.cuda.synchronize()
    mine = mine.cpu().numpy().view(np.uint32)
    ref = ref.cpu().numpy().view(np.uint32)
    assert np.array_equal(mine, ref), "device Philox4x32-10 differs from cuRAND's"
    for i in range(0, n, 97):
        assert np.array_equal(mine[i], orc.philox4x32_10(ctr[i], key[i]))
    assert list(mine[0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]


def test_e4m3_hardware_sr_pairs_match_oracle(P, orc):
    """The conversion unit's stochastic rounding, as the requant kernels use it: value pair
    (even, odd) with one random word, even rounded with its low half, odd with its high half,
    the two other result bytes zero. Grid points, midpoints, the subnormal range, 448."""
    rng = np.random.default_rng(4)
    x = e4m3_inputs(rng)
    x = x[np.abs(x) <= 448.0]
    x = rng.permutation(x)
    x = x[: len(x) // 2 * 2]
    n = len(x) // 2
    rb = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    rb[:40] = [0, 0xFFFFFFFF, 0x0000FFFF, 0xFFFF0000, 0x80008000, 0x00010001, 0xFFFEFFFE, 0x7FFF8000] * 5
    xd = torch.from_numpy(x).cuda()
    rd = torch.from_numpy(rb.view(np.int32)).cuda()
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    assert P.probe_e4m3x2_sr_hw(_p(xd), _p(rd), _p(out), n, _stream()) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    lib = orc.lib()
    sr = lib.orc_e4m3_encode_sr
    want_even = np.fromiter((sr(float(v), int(k) & 0xFFFF) for v, k in zip(x[0::2], rb)), np.uint32, count=n)
    want_odd = np.fromiter((sr(float(v), int(k) >> 16) for v, k in zip(x[1::2], rb)), np.uint32, count=n)
    assert_bytes_equal((got & 0xFF).astype(np.uint8), want_even.astype(np.uint8), "hw SR byte 0 (even)")
    assert_bytes_equal(((got >> 16) & 0xFF).astype(np.uint8), want_odd.astype(np.uint8), "hw SR byte 2 (odd)")
    assert not np.any(got & 0xFF00FF00), "hw SR: unused result bytes not zero"


@pytest.mark.parametrize("s_dec", [1.0, 0.0123456789, 3.0e-30, 7.5e20])
def test_dequant8_f16_path_matches_oracle(P, orc, s_dec):
    """E2M1 x E4M3 x fp32 through the f16x2 conversion path equals the definition
    (exact product of the two decoded values, then one fp32 rounding), signed zeros included."""
    rng = np.random.default_rng(5)
    scales = np.array([c for c in range(256) if (c & 0x7F) != 0x7F] * 16, dtype=np.uint8)
    n = len(scales)
    words = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    words[:2] = [0x76543210, 0xFEDCBA98]          # every code once
    wd = torch.from_numpy(words.view(np.int32)).cuda()
    sd = torch.from_numpy(scales).cuda()
    f16 = torch.empty(8 * n, dtype=torch.float32, device="cuda")
    ref = torch.empty_like(f16)
    assert P.probe_dequant8(_p(wd), _p(sd), ctypes.c_float(s_dec), _p(f16), _p(ref), n, _stream()) == 0
    torch.cuda.synchronize()
    e2 = np.array([orc.e2m1_decode(c) for c in range(16)], dtype=np.float64)
    e4 = np.array([orc.e4m3_decode(c) if (c & 0x7F) != 0x7F else 0.0 for c in range(256)], dtype=np.float64)
    codes = (words[:, None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
    prod = e2[codes] * e4[scales][:, None]                # exact in fp64
    want = (prod.astype(np.float32) * np.float32(s_dec)).astype(np.float32).reshape(-1)
    got = f16.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "f16x2 dequant differs from the definition"
    assert np.array_equal(got.view(np.uint32), ref.cpu().numpy().view(np.uint32))
