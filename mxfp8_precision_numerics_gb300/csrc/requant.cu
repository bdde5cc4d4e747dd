// requant.cu — dequantize -> [transpose] -> [16-point RHT] -> MXFP8 with stochastic rounding,
// and the stand-alone 16-point random Hadamard transform.
//
// 4bit.vizuara.ai §9-10: the saved NVFP4 tensors are dequantized, transposed and
// re-quantized to MXFP8 with stochastic rounding (E[w_q] = E[(w_q^T)^T]); the output gradient
// is quantized to MXFP8 twice, as it is for dgrad and transposed for wgrad.
// "Pretraining Large Language Models with NVFP4", "Random Hadamard Transforms": the wgrad
// operands are rotated along the contraction dimension in groups of 16.
// "FP4 Training on Blackwell", "The scaling math, worked": power-of-two block scale
// 2^ceil(log2(amax / vmax)), here with vmax = 448 (E4M3).
//
// Kernels
//   requant_rows_kernel  (transpose = 0): one thread per 32-value output block, read
//                        straight from HBM (bf16: 64 B, NVFP4: 16 B codes + 2 scales).
//   requant_t_kernel     (transpose = 1): a CTA dequantizes a 64 x 64 input tile into shared
//                        memory (fp32, padded rows), then each thread reads one input column
//                        segment of 32 = one output block, transforms, quantizes and writes
//                        32 bytes of the output row.
#include "fp4q_common.cuh"
#include "fp4q_internal.h"

namespace fp4q {

// Quantize 32 fp32 values (one MXFP8 block) and store 32 E4M3 bytes + 1 E8M0 byte.
// kRht: the block is two transform groups whose sign flips the caller has already applied;
// the butterflies and the 1/4 scaling happen here.
template <bool kRht, bool kSR>
__device__ __forceinline__ void mx_encode_block(float (&v)[32], uint64_t seed, uint32_t tag,
                                                uint64_t out_idx0, uint8_t* __restrict__ out32,
                                                uint8_t* __restrict__ out_sc) {
    if (kRht) {
        fwht16_quarter(v);
        fwht16_quarter(v + 16);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_exponent(amax);
    const float inv = exp2i(-e);
    uint32_t words[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        float t[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) t[j] = __fmul_rn(v[8 * g + j], inv);
        if (kSR) {
            // element 8g+j draws the low (j even) or high (j odd) half of word j/2
            const uint4 r = sr_block8(seed, tag, (out_idx0 >> 3) + (uint64_t)g);
            words[2 * g] = __byte_perm(e4m3x2_sr_hw(t[0], t[1], r.x), e4m3x2_sr_hw(t[2], t[3], r.y), 0x6420);
            words[2 * g + 1] = __byte_perm(e4m3x2_sr_hw(t[4], t[5], r.z), e4m3x2_sr_hw(t[6], t[7], r.w), 0x6420);
        } else {
            words[2 * g] = e4m3x4_rn_hw(t[0], t[1], t[2], t[3]);
            words[2 * g + 1] = e4m3x4_rn_hw(t[4], t[5], t[6], t[7]);
        }
    }
    uint4* o = reinterpret_cast<uint4*>(out32);
    __stcs(o, make_uint4(words[0], words[1], words[2], words[3]));
    __stcs(o + 1, make_uint4(words[4], words[5], words[6], words[7]));
    *out_sc = (uint8_t)(e + 127);
}

// Two bf16 values of one 32-bit word -> fp32 (exact).
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float* out) {
    out[0] = bf16_to_f32(w & 0xFFFFu);
    out[1] = __uint_as_float(w & 0xFFFF0000u);
}

// ---------------------------------------------------------------------------------------
// transpose = 0
// ---------------------------------------------------------------------------------------
template <int kKind, bool kRht, bool kSR>
__global__ void __launch_bounds__(256) requant_rows_kernel(RequantArgs a) {
    const int64_t nb = a.cols >> 5;
    const int64_t total = a.rows * nb;
    const float s_dec = (kKind == 0) ? 1.0f : *a.in_s_dec;
    // sign masks of the transform positions, packed like the input words
    uint32_t bm[8], nm0 = 0, nm1 = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) bm[p] = kRht ? bf16_sign_mask2(a.rht_signs, 2 * p) : 0u;
    if (kRht) {
        nm0 = e2m1_sign_mask8(a.rht_signs, 0);
        nm1 = e2m1_sign_mask8(a.rht_signs, 8);
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total; b += stride) {
        const int64_t r = b / nb, j = b - r * nb;
        float v[32];
        if (kKind == 0) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(a.in) + r * a.cols + j * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 p = __ldcs(src + q);
                uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) bf16x2_to_f32(w[k] ^ bm[4 * (q & 1) + k], v + 8 * q + 2 * k);
            }
        } else {
            const uint4 c = __ldcs(reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(a.in) + r * (a.cols >> 1) + j * 16));
            uint32_t s0, s1;
            if (kKind == 1) {
                s0 = a.in_scales[r * (a.cols >> 4) + 2 * j];
                s1 = a.in_scales[r * (a.cols >> 4) + 2 * j + 1];
            } else {
                s0 = a.in_scales[(r >> 4) * (a.cols >> 4) + 2 * j];
                s1 = a.in_scales[(r >> 4) * (a.cols >> 4) + 2 * j + 1];
            }
            const uint32_t f0 = e4m3_to_f16x2_dup(s0), f1 = e4m3_to_f16x2_dup(s1);
            dequant8_f16(c.x ^ nm0, f0, s_dec, v);
            dequant8_f16(c.y ^ nm1, f0, s_dec, v + 8);
            dequant8_f16(c.z ^ nm0, f1, s_dec, v + 16);
            dequant8_f16(c.w ^ nm1, f1, s_dec, v + 24);
        }
        mx_encode_block<kRht, kSR>(v, a.seed, a.tag, (uint64_t)(r * a.cols + j * 32),
                                   a.out_e4m3 + r * a.cols + j * 32, a.out_e8m0 + b);
    }
}

// ---------------------------------------------------------------------------------------
// transpose = 1: 64 x 64 input tile per CTA, 128 threads. The transform groups run along
// the input's rows (the output's contiguous dimension), so the sign of input row r is
// that of position r mod 16 and is applied to whole packed words at load time.
// ---------------------------------------------------------------------------------------
constexpr int kTR = 64, kTC = 64, kPad = 1;

template <int kKind, bool kRht, bool kSR>
__global__ void __launch_bounds__(128) requant_t_kernel(RequantArgs a) {
    __shared__ float tile[kTR][kTC + kPad];
    const int64_t r0 = (int64_t)blockIdx.y * kTR;   // input rows   = output columns
    const int64_t c0 = (int64_t)blockIdx.x * kTC;   // input columns = output rows
    const int tid = threadIdx.x;

    // ---- load + dequantize into shared memory (row-major, input orientation)
    if (kKind == 0) {
        const uint16_t* in = static_cast<const uint16_t*>(a.in);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = tid + 128 * i;          // 512 vectors of 8 bf16
            const int rr = v >> 3, cc = (v & 7) * 8;
            float* dst = &tile[rr][cc];
            if (r0 + rr < a.rows && c0 + cc < a.cols) {
                const uint32_t m = kRht ? ((a.rht_signs >> (rr & 15)) & 1u) * 0x80008000u : 0u;
                uint4 p = __ldcs(reinterpret_cast<const uint4*>(in + (r0 + rr) * a.cols + c0 + cc));
                bf16x2_to_f32(p.x ^ m, dst);
                bf16x2_to_f32(p.y ^ m, dst + 2);
                bf16x2_to_f32(p.z ^ m, dst + 4);
                bf16x2_to_f32(p.w ^ m, dst + 6);
            }
        }
    } else {
        const int rr = tid >> 1, half = tid & 1;
        const int64_t gr = r0 + rr, gc = c0 + 32 * half;
        if (gr < a.rows && gc < a.cols) {
            const float s_dec = *a.in_s_dec;
            const uint32_t m = kRht ? ((a.rht_signs >> (rr & 15)) & 1u) * 0x88888888u : 0u;
            const uint4 c = __ldcs(reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(a.in) + gr * (a.cols >> 1) + (gc >> 1)));
            uint32_t s0, s1;
            if (kKind == 1) {
                s0 = a.in_scales[gr * (a.cols >> 4) + (gc >> 4)];
                s1 = a.in_scales[gr * (a.cols >> 4) + (gc >> 4) + 1];
            } else {
                s0 = a.in_scales[(gr >> 4) * (a.cols >> 4) + (gc >> 4)];
                s1 = a.in_scales[(gr >> 4) * (a.cols >> 4) + (gc >> 4) + 1];
            }
            const uint32_t f0 = e4m3_to_f16x2_dup(s0), f1 = e4m3_to_f16x2_dup(s1);
            float* dst = &tile[rr][32 * half];
            dequant8_f16(c.x ^ m, f0, s_dec, dst);
            dequant8_f16(c.y ^ m, f0, s_dec, dst + 8);
            dequant8_f16(c.z ^ m, f1, s_dec, dst + 16);
            dequant8_f16(c.w ^ m, f1, s_dec, dst + 24);
        }
    }
    __syncthreads();

    // ---- one output block per thread: output row c0 + c, output columns r0 + 32*blk + [0, 32)
    const int c = tid & 63, blk = tid >> 6;
    const int64_t orow = c0 + c, ocol = r0 + 32 * blk;
    if (orow < a.cols && ocol < a.rows) {
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = tile[32 * blk + k][c];
        const int64_t oidx = orow * a.rows + ocol;
        mx_encode_block<kRht, kSR>(v, a.seed, a.tag, (uint64_t)oidx,
                                   a.out_e4m3 + oidx, a.out_e8m0 + (oidx >> 5));
    }
}

// ---------------------------------------------------------------------------------------
// stand-alone RHT16: one thread per group of 16
// ---------------------------------------------------------------------------------------
template <bool kBf16>
__global__ void __launch_bounds__(256) rht16_kernel(const void* __restrict__ in, float* __restrict__ out,
                                                    int64_t groups, uint32_t signs) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        float v[16];
        if (kBf16) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(in) + g * 16);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint4 p = __ldcs(src + q);
                uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * q + 2 * k] = bf16_to_f32(w[k] & 0xFFFFu);
                    v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
                }
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(in) + g * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 p = __ldcs(src + q);
                v[4 * q] = p.x; v[4 * q + 1] = p.y; v[4 * q + 2] = p.z; v[4 * q + 3] = p.w;
            }
        }
        rht16_inplace(v, signs);
        float4* dst = reinterpret_cast<float4*>(out + g * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) __stcs(dst + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    }
}

// ---------------------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------------------
template <int kKind, bool kRht, bool kSR>
static void launch_requant_t(const RequantArgs& a, cudaStream_t st) {
    if (a.transpose) {
        dim3 grid((unsigned)((a.cols + kTC - 1) / kTC), (unsigned)((a.rows + kTR - 1) / kTR));
        requant_t_kernel<kKind, kRht, kSR><<<grid, 128, 0, st>>>(a);
    } else {
        int64_t items = a.rows * (a.cols / 32);
        int64_t g = (items + 255) / 256;
        const int64_t cap = (int64_t)num_sms() * 8;
        if (g > cap) g = cap;
        requant_rows_kernel<kKind, kRht, kSR><<<(unsigned)(g < 1 ? 1 : g), 256, 0, st>>>(a);
    }
}

template <int kKind>
static void launch_requant_k(const RequantArgs& a, cudaStream_t st) {
    if (a.rht) {
        if (a.rounding) launch_requant_t<kKind, true, true>(a, st);
        else launch_requant_t<kKind, true, false>(a, st);
    } else {
        if (a.rounding) launch_requant_t<kKind, false, true>(a, st);
        else launch_requant_t<kKind, false, false>(a, st);
    }
}

cudaError_t launch_requant(const RequantArgs& a, cudaStream_t st) {
    switch (a.in_kind) {
        case 0: launch_requant_k<0>(a, st); break;
        case 1: launch_requant_k<1>(a, st); break;
        default: launch_requant_k<2>(a, st); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_rht16(const void* in, int in_is_bf16, float* out, int64_t rows, int64_t cols,
                         uint32_t signs, cudaStream_t st) {
    const int64_t groups = rows * (cols / 16);
    int64_t g = (groups + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    if (in_is_bf16) rht16_kernel<true><<<(unsigned)(g < 1 ? 1 : g), 256, 0, st>>>(in, out, groups, signs);
    else rht16_kernel<false><<<(unsigned)(g < 1 ? 1 : g), 256, 0, st>>>(in, out, groups, signs);
    return cudaGetLastError();
}

}  // namespace fp4q
