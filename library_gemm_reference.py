"""cuBLASLt's block-scaled GEMMs on this GPU, as a reference point for the library's own kernels:
MXFP8 (E4M3 with E8M0 per 32) and NVFP4 (E2M1 with E4M3 per 16) through torch._scaled_mm, and a
bf16 torch.mm, at the shapes the benchmark times. A measurement tool, not part of the library (the
library's GEMMs are its own tcgen05 kernels). Operand and scale values are arbitrary: the timing
does not depend on them.

    python library_gemm_reference.py
"""
import torch


def rup(x, m):
    return (x + m - 1) // m * m


def timeit(fn, flops, name, reps=20):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    med = ts[len(ts) // 2]
    print(f"{name:44s} median {med * 1e3:9.1f} us  {flops / (med * 1e-3) / 1e12:8.1f} TFLOP/s", flush=True)


def main():
    dev = "cuda"
    print("torch", torch.__version__, torch.cuda.get_device_name(), flush=True)
    for (M, N, K) in [(16384, 14336, 4096), (16384, 16384, 4096), (16384, 4096, 16384), (32768, 32768, 8192)]:
        fl = 2.0 * M * N * K
        a = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
        b = torch.randn(N, K, device=dev, dtype=torch.bfloat16)
        timeit(lambda: torch.mm(a, b.t()), fl, f"bf16 mm {M}x{N}x{K}")
        del a, b
        # MXFP8: scales sized for cuBLASLt's 128 x 4 blocked layout
        a = torch.randint(0, 0x7E, (M, K), device=dev, dtype=torch.uint8).view(torch.float8_e4m3fn)
        b = torch.randint(0, 0x7E, (N, K), device=dev, dtype=torch.uint8).view(torch.float8_e4m3fn)
        sa = torch.full((rup(M, 128) * rup(K // 32, 4),), 127, device=dev, dtype=torch.uint8).view(torch.float8_e8m0fnu)
        sb = torch.full((rup(N, 128) * rup(K // 32, 4),), 127, device=dev, dtype=torch.uint8).view(torch.float8_e8m0fnu)
        timeit(lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16), fl, f"mxfp8 _scaled_mm {M}x{N}x{K}")
        del a, b, sa, sb
        # NVFP4: two E2M1 codes per byte, E4M3 scales per 16
        a = torch.randint(0, 256, (M, K // 2), device=dev, dtype=torch.uint8).view(torch.float4_e2m1fn_x2)
        b = torch.randint(0, 256, (N, K // 2), device=dev, dtype=torch.uint8).view(torch.float4_e2m1fn_x2)
        sa = torch.full((rup(M, 128) * rup(K // 16, 4),), 0x38, device=dev, dtype=torch.uint8).view(torch.float8_e4m3fn)
        sb = torch.full((rup(N, 128) * rup(K // 16, 4),), 0x38, device=dev, dtype=torch.uint8).view(torch.float8_e4m3fn)
        timeit(lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16), fl, f"nvfp4 _scaled_mm {M}x{N}x{K}")
        del a, b, sa, sb
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
