"""Seeded synthetic inputs for the NVFP4 linear layer (no quantization arithmetic here).

Shared by the tests, the benchmark and the smoke check; it feeds both the CUDA
library and the CPU oracle the same bf16 bytes. Every tensor is generated on the
CPU with ``torch.Generator`` and a fixed seed, then cast to bf16.

Distributions (shapes of GPT / MoE linear layers, as the pages' workloads):
  * activations X: N(0, 1) with exactly floor(0.001 * numel) distinct positions,
    drawn uniformly without replacement, multiplied by 50 before the bf16 cast;
  * weights W: N(0, 0.02);
  * output gradients dY: Student-t with 3 degrees of freedom times 1e-3, built as
    Z / sqrt(chi2_3 / 3) with chi2_3 the sum of three squared standard normals.
Random numbers the method itself consumes (the stochastic-rounding seed, the
Hadamard sign mask, the MoE routing) are drawn here too and passed in as inputs.
"""
import math

import torch

# The five workloads: name -> shapes. M = tokens, K = in features, N = out features.
CONFIGS = {
    "linear_fwd_256x512": dict(M=256, K=512, N=256, seed=0),
    "moe_expert_fwd_8x1024x1536x4096": dict(E=8, T=8192, K=4096, N=1536, seed=1),
    "backward_requant_8192x4096x4096": dict(M=8192, K=4096, N=4096, seed=2),
    "wq2d_gemm_sweep_14336x4096": dict(N=14336, K=4096, Ms=(1024, 4096, 16384), seed=3),
    "gpt_mlp_fwd_bwd_16384x4096x16384": dict(M=16384, D=4096, F=16384, seed=4),
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(rows: int, cols: int, seed: int, std: float = 1.0) -> torch.Tensor:
    g = generator(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_with_outliers(rows: int, cols: int, seed: int, std: float = 1.0,
                         frac: float = 1e-3, mult: float = 50.0) -> torch.Tensor:
    g = generator(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    n = x.numel()
    k = int(math.floor(frac * n))
    if k > 0:
        pos = torch.randperm(n, generator=g)[:k]
        flat = x.view(-1)
        flat[pos] = flat[pos] * mult
    return x.to(torch.bfloat16)


def student_t(rows: int, cols: int, seed: int, df: int = 3, scale: float = 1e-3) -> torch.Tensor:
    g = generator(seed)
    z = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    chi2 = torch.zeros(rows, cols, dtype=torch.float32)
    for _ in range(df):
        c = torch.randn(rows, cols, generator=g, dtype=torch.float32)
        chi2.addcmul_(c, c)
    t = z / torch.sqrt(chi2 / df)
    return (t * scale).to(torch.bfloat16)


def routing(tokens: int, experts: int, seed: int):
    """Uniform top-1 routing: a seeded permutation of the tokens split into equal
    groups. Returns (perm, row_offsets) with row_offsets of length experts + 1."""
    g = generator(seed)
    perm = torch.randperm(tokens, generator=g)
    per = tokens // experts
    offs = torch.arange(0, experts + 1, dtype=torch.int32) * per
    return perm, offs


def rht_signs(seed: int) -> int:
    """A 16-bit random sign mask for the Hadamard transform (bit i set -> negate i)."""
    g = generator(seed + 0x5EED)
    return int(torch.randint(0, 1 << 16, (1,), generator=g).item())


def sr_seed(seed: int) -> int:
    """A 64-bit key for the stochastic-rounding generator."""
    g = generator(seed + 0xC0FFEE)
    hi = int(torch.randint(0, 1 << 31, (1,), generator=g).item())
    lo = int(torch.randint(0, 1 << 31, (1,), generator=g).item())
    return (hi << 32) | lo


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
