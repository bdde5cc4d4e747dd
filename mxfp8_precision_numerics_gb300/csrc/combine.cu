// combine.cu — the MoE combine wire format: RHT32 + block-scaled S2F6, encode and decode.
//
// 4bit.vizuara.ai §11 ("Combine is harder"): a layer output is rotated 32 values at a time
// (sign flips by a fixed pattern, then the 32 sums and differences, each over sqrt 32) and
// sent as S2F6, a signed 8-bit integer over 64, with one power-of-two scale per 32 values
// (8.25 bits per value); the receiver dequantizes and adds the arrivals, then undoes the
// rotation. "End-to-End 4-Bit Training" (Thinking Machines), 合并阶段: RHT32, S2F6 with an
// E8M0 scale per 32, decoded and aggregated on arrival, then the inverse transform. The
// arithmetic is in fp4q_common.cuh (rht32_forward / rht32_inverse / s2f6_encode32 /
// s2f6_decode4); the same encoder also runs inside the GEMM epilogue (gemm.cu).
//
// Kernels (both HBM streams, one thread per group of 32 values, grid-stride):
//   combine_encode_kernel  fp32 or bf16 [rows][cols] -> S2F6 bytes [rows][cols] + E8M0 [rows][cols/32]
//   combine_decode_kernel  k arrivals per token (rows t*k .. t*k+k-1) -> their sum rotated back,
//                          fp32 or bf16 [tokens][cols]
// The conversion instructions for block-scaled S2F6 that the pages list are not accepted by
// this toolkit's assembler for sm_103a; the values are rounded with cvt.rni to int32 instead.
#include <cuda_bf16.h>

#include "fp4q_common.cuh"
#include "fp4q_internal.h"

namespace fp4q {

template <bool kBf16>
__global__ void __launch_bounds__(256) combine_encode_kernel(const void* __restrict__ in, int64_t groups,
                                                             uint32_t signs, uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ e8m0) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        float v[32];
        if (kBf16) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(in) + g * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 p = __ldg(src + q);
                const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * q + 2 * k] = __uint_as_float(w[k] << 16);
                    v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
                }
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(in) + g * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 p = __ldg(src + q);
                v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
            }
        }
        rht32_forward(v, signs);
        uint32_t out[8];
        const uint32_t sc = s2f6_encode32(v, out);
        uint4* dst = reinterpret_cast<uint4*>(codes + g * 32);
        __stcs(dst, make_uint4(out[0], out[1], out[2], out[3]));
        __stcs(dst + 1, make_uint4(out[4], out[5], out[6], out[7]));
        e8m0[g] = (uint8_t)sc;
    }
}

template <bool kOutBf16>
__global__ void __launch_bounds__(256) combine_decode_kernel(const uint8_t* __restrict__ codes,
                                                             const uint8_t* __restrict__ e8m0,
                                                             int64_t tokens, int64_t k, int64_t gpr,
                                                             uint32_t signs, void* __restrict__ out) {
    const int64_t groups = tokens * gpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const int64_t t = g / gpr, c = g - t * gpr;
        float acc[32];
        for (int64_t j = 0; j < k; ++j) {            // arrivals in slot order
            const int64_t src = (t * k + j) * gpr + c;
            const uint4* cp = reinterpret_cast<const uint4*>(codes + src * 32);
            const uint4 a = __ldcs(cp), b = __ldcs(cp + 1);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            const uint32_t sc = e8m0[src];
            float z[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) s2f6_decode4(w[q], sc, z + 4 * q);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = j == 0 ? z[i] : __fadd_rn(acc[i], z[i]);
        }
        rht32_inverse(acc, signs);
        if (kOutBf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + g * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * q + 2 * m], acc[8 * q + 2 * m + 1]);
                    w[m] = *reinterpret_cast<const uint32_t*>(&h);
                }
                __stcs(dst + q, make_uint4(w[0], w[1], w[2], w[3]));
            }
        } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + g * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                __stcs(dst + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
        }
    }
}

static unsigned combine_grid(int64_t groups) {
    int64_t g = (groups + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

cudaError_t launch_combine_encode(const void* in, int in_bf16, int64_t rows, int64_t cols, uint32_t signs,
                                  uint8_t* codes, uint8_t* e8m0, cudaStream_t st) {
    const int64_t groups = rows * (cols / 32);
    if (in_bf16)
        combine_encode_kernel<true><<<combine_grid(groups), 256, 0, st>>>(in, groups, signs, codes, e8m0);
    else
        combine_encode_kernel<false><<<combine_grid(groups), 256, 0, st>>>(in, groups, signs, codes, e8m0);
    return cudaGetLastError();
}

cudaError_t launch_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k,
                                  int64_t cols, uint32_t signs, void* out, int out_bf16, cudaStream_t st) {
    const int64_t gpr = cols / 32;
    const unsigned g = combine_grid(tokens * gpr);
    if (out_bf16)
        combine_decode_kernel<true><<<g, 256, 0, st>>>(codes, e8m0, tokens, k, gpr, signs, out);
    else
        combine_decode_kernel<false><<<g, 256, 0, st>>>(codes, e8m0, tokens, k, gpr, signs, out);
    return cudaGetLastError();
}

}  // namespace fp4q
