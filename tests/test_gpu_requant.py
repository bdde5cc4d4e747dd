"""fp4q_requant_t_mxfp8_sr and fp4q_rht16 against the oracle, bit for bit: every input
kind x transpose x RHT x rounding mode on ragged tile shapes, and sampled output rows
of the full-size backward tensors (dY 8192x4096, X_q 8192x4096, W_q 4096x4096)."""
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


def make_input(F, orc, kind, rows, cols, seed):
    """-> (device input, device scales, device s_dec, oracle data, oracle scales, oracle s_dec)."""
    if kind == F.IN_BF16:
        x = I.student_t(rows, cols, seed=seed)
        return x.cuda(), None, None, I.bf16_bits(x), None, 1.0
    x = I.normal_with_outliers(rows, cols, seed=seed)
    xb = I.bf16_bits(x)
    if kind == F.IN_NVFP4_1D:
        oc, os_, _, osd = orc.quantize_1d(xb)
    else:
        oc, os_, _, osd = orc.quantize_2d(xb)
    return (torch.from_numpy(oc).cuda(), torch.from_numpy(os_).cuda(),
            torch.tensor([osd], dtype=torch.float32, device="cuda"), oc, os_, osd)


CASES = [(k, t, r, m) for k in (0, 1, 2) for t in (0, 1) for r in (0, 1) for m in (0, 1)]


@pytest.mark.parametrize("kind,transpose,rht,rounding", CASES)
def test_requant_all_modes_ragged(F, orc, kind, transpose, rht, rounding):
    rows, cols = 96, 160          # 64-row tiles + a ragged 32-row tail; 64,64,32 columns
    seed, signs, tag = 0x1234_5678_9ABC_DEF0, 0xA5C3, 7
    din, dsc, dsd, oin, osc, osd = make_input(F, orc, kind, rows, cols, seed=kind * 10 + 1)
    e4, e8 = F.requant_mxfp8(kind, din, dsc, dsd, rows, cols, transpose, rht, signs, rounding, seed, tag)
    torch.cuda.synchronize()
    r4, r8 = orc.requant_mxfp8(kind, oin, osc, osd, rows, cols, transpose, rht, signs, rounding, seed, tag)
    what = f"kind={kind} T={transpose} rht={rht} sr={rounding}"
    assert_bytes_equal(e8.cpu().numpy(), r8, what + " e8m0")
    assert_bytes_equal(e4.cpu().numpy(), r4, what + " e4m3")


def test_requant_seed_and_tag_change_the_draws(F, orc):
    din, dsc, dsd, *_ = make_input(F, orc, F.IN_BF16, 64, 64, seed=3)
    a, _ = F.requant_mxfp8(0, din, dsc, dsd, 64, 64, 1, 0, 0, F.SR, 1, 3)
    b, _ = F.requant_mxfp8(0, din, dsc, dsd, 64, 64, 1, 0, 0, F.SR, 2, 3)
    c, _ = F.requant_mxfp8(0, din, dsc, dsd, 64, 64, 1, 0, 0, F.SR, 1, 4)
    d, _ = F.requant_mxfp8(0, din, dsc, dsd, 64, 64, 1, 0, 0, F.SR, 1, 3)
    assert torch.equal(a, d)                       # deterministic for a fixed (seed, tag)
    assert not torch.equal(a, b) and not torch.equal(a, c)


def test_requant_sr_is_unbiased_on_device(F, orc):
    """The mean of many SR requants of W_q^T approaches the dequantized W_q^T."""
    w = I.normal(64, 128, seed=12, std=0.02)
    oc, ot, _, osd = orc.quantize_2d(I.bf16_bits(w))
    xq_t = orc.dequant_nvfp4(oc, ot, 2, osd).T
    c, t, sd = torch.from_numpy(oc).cuda(), torch.from_numpy(ot).cuda(), torch.tensor([osd], device="cuda")
    k = 256
    acc = np.zeros_like(xq_t)
    for s in range(k):
        e4, e8 = F.requant_mxfp8(F.IN_NVFP4_2D, c, t, sd, 64, 128, 1, 0, 0, F.SR, s, F.TAG_WT)
        acc += orc.dequant_mxfp8(e4.cpu().numpy(), e8.cpu().numpy())
    err = np.linalg.norm(acc / k - xq_t) / np.linalg.norm(xq_t)
    e4, e8 = F.requant_mxfp8(F.IN_NVFP4_2D, c, t, sd, 64, 128, 1, 0, 0, F.SR, 0, F.TAG_WT)
    one = np.linalg.norm(orc.dequant_mxfp8(e4.cpu().numpy(), e8.cpu().numpy()) - xq_t) / np.linalg.norm(xq_t)
    assert err < 2 * one / np.sqrt(k)


def _sample_rows(n, k=48, seed=0):
    rng = np.random.default_rng(seed)
    head = list(range(0, 16))
    tail = list(range(n - 16, n))
    mid = sorted(rng.choice(np.arange(16, n - 16), k - 32, replace=False).tolist())
    return head + mid + tail


def check_sampled(F, orc, kind, din, dsc, dsd, oin, osc, osd, rows, cols, transpose, rht, signs, seed, tag, what):
    e4, e8 = F.requant_mxfp8(kind, din, dsc, dsd, rows, cols, transpose, rht, signs, F.SR, seed, tag)
    torch.cuda.synchronize()
    orows = cols if transpose else rows
    e4 = e4.cpu().numpy()
    e8 = e8.cpu().numpy()
    for r in _sample_rows(orows):
        r4, r8 = orc.requant_mxfp8(kind, oin, osc, osd, rows, cols, transpose, rht, signs, F.SR, seed, tag,
                                   out_rows=(r, r + 1))
        assert_bytes_equal(e8[r:r + 1], r8, f"{what} e8m0 row {r}")
        assert_bytes_equal(e4[r:r + 1], r4, f"{what} e4m3 row {r}")
    # every block's max lands in (224, 448] (ceiling exponent) unless the block is zero
    vals = orc.dequant_mxfp8(e4[:64], e8[:64])
    t = np.abs(vals).reshape(64, -1, 32).max(axis=2) / 2.0 ** (e8[:64].astype(np.int64) - 127)
    assert np.all((t == 0) | ((t > 200) & (t <= 448)))


def test_backward_requant_full_size_sampled(F, orc):
    M, K, N = 8192, 4096, 4096
    seed, signs = I.sr_seed(2), I.rht_signs(2)
    dy = I.student_t(M, N, seed=2)
    dyd, dyb = dy.cuda(), I.bf16_bits(dy)
    check_sampled(F, orc, 0, dyd, None, None, dyb, None, 1.0, M, N, 0, 0, 0, seed, F.TAG_DY_ROWS, "dY rows")
    check_sampled(F, orc, 0, dyd, None, None, dyb, None, 1.0, M, N, 1, 1, signs, seed, F.TAG_DY_T, "dY^T rht")
    x = I.normal_with_outliers(M, K, seed=22)
    oc, os_, _, osd = orc.quantize_1d(I.bf16_bits(x))
    check_sampled(F, orc, 1, torch.from_numpy(oc).cuda(), torch.from_numpy(os_).cuda(),
                  torch.tensor([osd], device="cuda"), oc, os_, osd, M, K, 1, 1, signs, seed, F.TAG_XT, "X_q^T rht")
    w = I.normal(N, K, seed=23, std=0.02)
    wc, wt, _, wsd = orc.quantize_2d(I.bf16_bits(w))
    check_sampled(F, orc, 2, torch.from_numpy(wc).cuda(), torch.from_numpy(wt).cuda(),
                  torch.tensor([wsd], device="cuda"), wc, wt, wsd, N, K, 1, 0, 0, seed, F.TAG_WT, "W_q^T")


@pytest.mark.parametrize("bf16", [False, True])
def test_rht16_matches_oracle(F, orc, bf16):
    rows, cols = 37, 272
    x = I.normal_with_outliers(rows, cols, seed=31)
    if bf16:
        xd, xo = x.cuda(), I.bf16_bits(x)
    else:
        xf = x.float() * 1.2345
        xd, xo = xf.cuda(), xf.numpy()
    out = F.rht16(xd, 0xBEEF)
    torch.cuda.synchronize()
    want = orc.rht16(xo, 0xBEEF, is_bf16=bf16)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("rows,cols,rht", [(64, 128, 1), (96, 160, 1), (256, 544, 0), (8192, 4096, 1)])
def test_requant_bf16_dual_equals_the_two_calls(F, orc, rows, cols, rht):
    """fp4q_requant_bf16_dual: the rowwise and the transposed (RHT) quantizations of the output
    gradient from one read are the two separate requantizations, byte for byte (ragged 64 x 128
    tiles included), and sampled rows match the oracle."""
    seed, signs = I.sr_seed(7), I.rht_signs(7)
    dy = I.student_t(rows, cols, seed=rows + cols)
    d = dy.cuda()
    (r4, r8), (t4, t8) = F.requant_bf16_dual(d, rht, signs, F.SR, seed, F.TAG_DY_ROWS, F.TAG_DY_T)
    g4, g8 = F.requant_mxfp8(F.IN_BF16, d, None, None, rows, cols, 0, 0, 0, F.SR, seed, F.TAG_DY_ROWS)
    u4, u8 = F.requant_mxfp8(F.IN_BF16, d, None, None, rows, cols, 1, rht, signs, F.SR, seed, F.TAG_DY_T)
    torch.cuda.synchronize()
    assert F.fp4q_device_status() == F.OK
    for got, want, what in ((r4, g4, "rows e4m3"), (r8, g8, "rows e8m0"), (t4, u4, "T e4m3"), (t8, u8, "T e8m0")):
        assert_bytes_equal(got.cpu().numpy(), want.cpu().numpy(), what)
    db = I.bf16_bits(dy)
    for b in (0, rows - 2):
        o4, o8 = orc.requant_mxfp8(0, db, None, 1.0, rows, cols, False, False, 0, orc.SR, seed, F.TAG_DY_ROWS,
                                   out_rows=(b, b + 2))
        assert_bytes_equal(r4[b:b + 2].cpu().numpy(), o4, "rows e4m3 vs oracle")
        assert_bytes_equal(r8[b:b + 2].cpu().numpy(), o8, "rows e8m0 vs oracle")
    for b in (0, cols - 2):
        o4, o8 = orc.requant_mxfp8(0, db, None, 1.0, rows, cols, True, bool(rht), signs, orc.SR, seed, F.TAG_DY_T,
                                   out_rows=(b, b + 2))
        assert_bytes_equal(t4[b:b + 2].cpu().numpy(), o4, "T e4m3 vs oracle")
        assert_bytes_equal(t8[b:b + 2].cpu().numpy(), o8, "T e8m0 vs oracle")
