"""Run one library call on a given shape repeatedly: a small, self-contained case for
profilers (e.g. ``ncu -k regex:gemm_pair_kernel -s 2 -c 1 python profile_case.py
--call gemm_mxfp8 --M 8192 --N 4096 --K 16384``). The commands of the summaries under
profiles/ run it.

Operands are random bytes of the right formats generated on the device (values do not
change the work any of these kernels does), so the case starts in seconds.
"""
import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from mxfp8_precision_numerics_gb300 import fp4q as F  # noqa: E402


def _e4m3(shape, g):
    c = torch.randint(0, 0x7E, shape, dtype=torch.uint8, device="cuda", generator=g)
    return c | (torch.randint(0, 2, shape, dtype=torch.uint8, device="cuda", generator=g) << 7)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--call", required=True,
                    choices=["gemm_mxfp8", "gemm_mxfp8_dgelu", "gemm_nvfp4", "gemm_nvfp4_gelu", "gemm_mxfp4", "quantize_1d",
                             "quantize_1d_given_amax", "quantize_2d", "requant_bf16_dual", "mlp_step",
                             "quantize_1d_rows46", "quantize_mxfp4", "requant_bf16_t_rht", "requant_bf16_rows",
                             "requant_nvfp4_t_rht", "requant_nvfp4_2d_t", "combine_encode", "combine_decode"])
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--K", type=int, default=16384)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--k", type=int, default=1, help="combine_decode: arrivals per token (M tokens)")
    ap.add_argument("--bf16", action="store_true", help="combine: bf16 encode input / decode output")
    ap.add_argument("--rht", action="store_true", help="quantize_mxfp4: rotate by RHT32 first")
    ap.add_argument("--f32", action="store_true", help="gemm_mxfp8: fp32 output (default bf16)")
    a = ap.parse_args()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    M, N, K = a.M, a.N, a.K
    if a.call == "gemm_mxfp8":
        A, B = _e4m3((M, K), g), _e4m3((N, K), g)
        As = torch.randint(120, 134, (M, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        Bs = torch.randint(120, 134, (N, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        fn = lambda: F.gemm_mxfp8(A, As, B, Bs, torch.float32 if a.f32 else torch.bfloat16)
    elif a.call == "gemm_mxfp8_dgelu":
        A, B = _e4m3((M, K), g), _e4m3((N, K), g)
        As = torch.randint(120, 134, (M, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        Bs = torch.randint(120, 134, (N, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        H = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
        fn = lambda: F.gemm_mxfp8_dgelu(A, As, B, Bs, H)
    elif a.call in ("gemm_nvfp4", "gemm_nvfp4_gelu"):
        A = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
        As = torch.randint(0x18, 0x58, (M, K // 16), dtype=torch.uint8, device="cuda", generator=g)
        Bs = torch.randint(0x18, 0x58, (N // 16, K // 16), dtype=torch.uint8, device="cuda", generator=g)
        one = torch.ones(1, device="cuda")
        if a.call == "gemm_nvfp4":
            fn = lambda: F.gemm_nvfp4(A, As, one, B, Bs, F.SCALE_2D, one, torch.bfloat16)
        else:
            fn = lambda: F.gemm_nvfp4_gelu(A, As, one, B, Bs, F.SCALE_2D, one)
    elif a.call == "gemm_mxfp4":
        A = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
        As = torch.randint(118, 136, (M, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        Bs = torch.randint(118, 136, (N, K // 32), dtype=torch.uint8, device="cuda", generator=g)
        fn = lambda: F.gemm_mxfp4(A, As, B, Bs, torch.bfloat16)
    elif a.call == "mlp_step":
        # the benchmark's step (tokens M, d_model N, ffn K): synthetic normal inputs on the device
        from mxfp8_precision_numerics_gb300 import layer
        x = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
        w1 = (torch.randn(K, N, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        w2 = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        dy = (torch.randn(M, N, device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
        fn = lambda: layer.mlp_step(x, w1, w2, dy, 12345, 0xA5C3)
    elif a.call == "combine_encode":
        y = torch.randn(M, K, device="cuda", generator=g)
        if a.bf16:
            y = y.to(torch.bfloat16)
        fn = lambda: F.combine_encode(y, 0x9E3779B9)
    elif a.call == "combine_decode":
        codes, e8 = F.combine_encode(torch.randn(M * a.k, K, device="cuda", generator=g), 0x9E3779B9)
        fn = lambda: F.combine_decode(codes, e8, a.k, 0x9E3779B9, torch.bfloat16 if a.bf16 else torch.float32)
    else:
        x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
        if a.call == "quantize_1d":
            fn = lambda: F.quantize_1d(x)
        elif a.call == "quantize_1d_given_amax":
            amax = x.float().abs().max().reshape(1)
            fn = lambda: F.quantize_1d(x, amax_in=amax)
        elif a.call == "requant_bf16_dual":
            fn = lambda: F.requant_bf16_dual(x, 1, 0xA5C3, F.SR, 1, 2, 3)
        elif a.call == "quantize_1d_rows46":
            fn = lambda: F.quantize_1d_rows(x, True)
        elif a.call == "quantize_mxfp4":
            fn = lambda: F.quantize_mxfp4(x, a.rht, 0x5EED1234)
        elif a.call == "quantize_2d":
            fn = lambda: F.quantize_2d(x)
        elif a.call == "requant_bf16_t_rht":
            fn = lambda: F.requant_mxfp8(F.IN_BF16, x, None, None, M, K, 1, 1, 0xA5C3, F.SR, 1, 3)
        elif a.call == "requant_bf16_rows":
            fn = lambda: F.requant_mxfp8(F.IN_BF16, x, None, None, M, K, 0, 0, 0, F.SR, 1, 2)
        else:
            c, s, d, _ = (F.quantize_1d(x) if a.call == "requant_nvfp4_t_rht" else F.quantize_2d(x))
            kind, rht = (F.IN_NVFP4_1D, 1) if a.call == "requant_nvfp4_t_rht" else (F.IN_NVFP4_2D, 0)
            fn = lambda: F.requant_mxfp8(kind, c, s, d, M, K, 1, rht, 0xA5C3, F.SR, 1, 4)
    for _ in range(a.reps):
        fn()
    torch.cuda.synchronize()
    st = F.fp4q_device_status()
    if st != F.OK:
        raise SystemExit("device status: " + F.status_str(st))
    print(f"{a.call} M={M} N={N} K={K} reps={a.reps}: ok")


if __name__ == "__main__":
    main()
