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
//   requant_t_kernel     (transpose = 1): persistent CTAs walk 64 x 128 input tiles, staged
//                        raw in shared memory one tile ahead; two lanes share one 32-value
//                        output block (one transform group each), see below.
// Input kinds: bf16; NVFP4 with 1D or 16x16 tile scales and one outer scale; NVFP4 with 1D
// scales and one outer scale per input row (the per-token activation form of
// 4bit.vizuara.ai §10), where each dequantized value takes its own row's s_dec.
#include "fp4q_common.cuh"
#include "fp4q_internal.h"

namespace fp4q {

// Quantize 32 fp32 values (one MXFP8 block) and store 32 E4M3 bytes + 1 E8M0 byte.
// kRht: the block is two transform groups whose sign flips the caller has already applied;
// the butterflies happen here. The transform's 1/4 is folded into the block's power-of-two
// scale, t = s * 2^(-e-2), which is the definition's fl(fl(s/4) * 2^-e) bit for bit whenever
// max|s| >= 2^-88: then every s with s/4 in the fp32 normal range gives the same single
// rounding of s * 2^(-e-2), and every smaller s gives |t| < 2^-27 under both orders, which
// rounds (to nearest or stochastically, U <= 1 - 2^-16) to a zero of the same sign.
// Blocks below that take the definition's order literally.
template <bool kRht, bool kSR>
__device__ __forceinline__ void mx_encode_block(float (&v)[32], uint64_t seed, uint32_t tag,
                                                uint64_t out_idx0, uint8_t* __restrict__ out32,
                                                uint8_t* __restrict__ out_sc) {
    if (kRht) {
        fwht16(v);
        fwht16(v + 16);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    int e;
    float inv;
    if (kRht) {
        e = mx_exponent(__fmul_rn(amax, 0.25f));        // max|s/4| = max|s| / 4 (monotone rounding)
        if (__float_as_uint(amax) >= 0x13800000u) {     // max|s| >= 2^-88
            inv = exp2i_wide(-e - 2);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], 0.25f);
            inv = exp2i(-e);
        }
    } else {
        e = mx_exponent(amax);
        inv = exp2i(-e);
    }
    uint32_t words[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        float t[8];
        mul8_f32x2(v + 8 * g, inv, t);
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
    const float s_dec_t = (kKind == 0 || kKind == 3) ? 1.0f : *a.in_s_dec;   // kind 3: per row
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
            const float s_dec = kKind == 3 ? a.in_s_dec[r] : s_dec_t;
            if (kKind != 2) {
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

// Half of an MXFP8 block: this lane's 16 values (one transform group), the other 16 in the
// partner lane (lane ^ 1); the block amax is combined with one shuffle. Same arithmetic as
// mx_encode_block. Every lane of the warp must call it (stores are predicated on `valid`).
// out_idx: output index of this lane's first value; out_sc: the block's E8M0 byte, written by
// the lane holding the first half (nullptr in the other).
template <bool kRht, bool kSR>
__device__ __forceinline__ void mx_encode_half(float (&v)[16], bool valid, uint64_t seed, uint32_t tag,
                                               uint64_t out_idx, uint8_t* __restrict__ out16,
                                               uint8_t* __restrict__ out_sc) {
    if (kRht) fwht16(v);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    int e;
    float inv;
    if (kRht) {
        e = mx_exponent(__fmul_rn(amax, 0.25f));
        if (__float_as_uint(amax) >= 0x13800000u) {     // max|s| >= 2^-88: fold the 1/4
            inv = exp2i_wide(-e - 2);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
            inv = exp2i(-e);
        }
    } else {
        e = mx_exponent(amax);
        inv = exp2i(-e);
    }
    uint32_t words[4];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        float t[8];
        mul8_f32x2(v + 8 * g, inv, t);
        if (kSR) {
            const uint4 r = sr_block8(seed, tag, (out_idx >> 3) + (uint64_t)g);
            words[2 * g] = __byte_perm(e4m3x2_sr_hw(t[0], t[1], r.x), e4m3x2_sr_hw(t[2], t[3], r.y), 0x6420);
            words[2 * g + 1] = __byte_perm(e4m3x2_sr_hw(t[4], t[5], r.z), e4m3x2_sr_hw(t[6], t[7], r.w), 0x6420);
        } else {
            words[2 * g] = e4m3x4_rn_hw(t[0], t[1], t[2], t[3]);
            words[2 * g + 1] = e4m3x4_rn_hw(t[4], t[5], t[6], t[7]);
        }
    }
    if (valid) {
        __stcs(reinterpret_cast<uint4*>(out16), make_uint4(words[0], words[1], words[2], words[3]));
        if (out_sc) *out_sc = (uint8_t)(e + 127);
    }
}

// ---------------------------------------------------------------------------------------
// transpose = 1. Persistent CTAs of 256 threads walk 64 x 128 input tiles; each tile's raw
// input (bf16 16 KB, or NVFP4 codes 4 KB) is brought into shared memory by cp.async one tile
// ahead, its block scales by plain loads one tile ahead. Thread (p, g) owns input columns 2p
// and 2p+1 of input rows 16g .. 16g+15: one transform group of one MXFP8 block of each of
// two output rows; one 32-bit word (bf16 pair) or one byte (E2M1 pair) per input row feeds
// both. Lanes 4p .. 4p+3 hold g = 0..3, so the two halves of a block sit in lanes l, l^1.
// Shared memory is XOR-swizzled by row group (bf16: 8 words, codes: 16 bytes, scales: 2
// entries) so that the four row groups reading one column pair hit distinct banks.
// The transform groups run along the input's rows (the output's contiguous dimension), so
// the sign of input row r is that of position r mod 16: for bf16 it is XORed onto the word,
// for NVFP4 it is folded into that row's block scale (E2M1 x (-scale) is exact).
// ---------------------------------------------------------------------------------------
constexpr int kTR = 64, kTC = 128, kTThreads = 256;

template <int kKind>
struct TStage {
    static constexpr uint32_t kBytes = kKind == 0 ? kTR * kTC * 2 : kTR * kTC / 2;   // 16 KB / 4 KB
};

// kDual (bf16 input): the same staged tile also gives the rowwise output (out2, tag2, no
// transform) — one read of the input for both of the output gradient's quantizations.
template <int kKind, bool kRht, bool kSR, bool kDual = false>
__global__ void __launch_bounds__(kTThreads) requant_t_kernel(RequantArgs a, int tiles_c, int n_tiles) {
    __shared__ __align__(16) uint8_t stage[2][TStage<kKind>::kBytes];
    __shared__ uint32_t sct[2][kKind == 0 ? 1 : kTR][8];   // per input row: f16x2 scales, signs folded
    __shared__ float sdr[2][kKind == 3 ? kTR : 1];          // kind 3: per input row outer scale
    const int tid = threadIdx.x;
    const int p = tid >> 2, grp = tid & 3, hb = grp & 1;
    const float s_dec = (kKind == 0 || kKind == 3) ? 1.0f : *a.in_s_dec;
    const int64_t sc_ld = a.cols >> 4;

    // cp.async of tile `tile` into buffer `buf`; block scales of the tile into `sreg`
    auto issue = [&](int tile, int buf, uint32_t (&sreg)[2], float& sdreg) {
        const int tr = tile / tiles_c, tc = tile - tr * tiles_c;
        const int64_t r0 = (int64_t)tr * kTR, c0 = (int64_t)tc * kTC;
        const uint32_t base = (uint32_t)__cvta_generic_to_shared(&stage[buf][0]);
        if (kKind == 0) {
            const uint16_t* in = static_cast<const uint16_t*>(a.in);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int ch = tid + kTThreads * i;          // 1024 chunks of 8 bf16 (4 words)
                const int row = ch >> 4, cw = (ch & 15) * 4;
                const bool ok = r0 + row < a.rows && c0 + 2 * cw < a.cols;
                const uint32_t dst = base + 4u * (uint32_t)(row * 64 + (cw ^ (8 * ((row >> 4) & 3))));
                cp_async16(dst, in + (ok ? (r0 + row) * a.cols + c0 + 2 * cw : 0), ok);
            }
        } else {
            const uint8_t* in = static_cast<const uint8_t*>(a.in);
            const int row = tid >> 2, cb = (tid & 3) * 16;   // 256 chunks of 32 codes
            const bool ok = r0 + row < a.rows && c0 + 2 * cb < a.cols;
            const uint32_t dst = base + (uint32_t)(row * 64 + (cb ^ (16 * ((row >> 4) & 3))));
            cp_async16(dst, in + (ok ? (r0 + row) * (a.cols >> 1) + (c0 >> 1) + cb : 0), ok);
            // block scale of each input row and block of 16 columns (2D: the row's 16 x 16 tile)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int idx = tid + kTThreads * i;
                const int srow = idx >> 3, blk = idx & 7;
                const int64_t grow = r0 + srow, gcol = (c0 >> 4) + blk;
                sreg[i] = 0;
                if (grow < a.rows && gcol < sc_ld)
                    sreg[i] = a.in_scales[(kKind == 2 ? (grow >> 4) : grow) * sc_ld + gcol];
            }
            if (kKind == 3 && tid < kTR) sdreg = r0 + tid < a.rows ? a.in_s_dec[r0 + tid] : 0.0f;
        }
        cp_async_commit();
    };

    int tile = blockIdx.x;
    if (tile >= n_tiles) return;
    uint32_t sreg[2] = {0, 0};
    float sdreg = 0.0f;
    issue(tile, 0, sreg, sdreg);
    for (int it = 0; tile < n_tiles; ++it, tile += gridDim.x) {
        const int buf = it & 1;
        if (kKind != 0) {
            // this tile's scales -> f16x2 (both halves), with the sign of the row's transform
            // position folded in
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int idx = tid + kTThreads * i;
                const int srow = idx >> 3, blk = idx & 7;
                uint32_t h = e4m3_to_f16x2_dup(sreg[i]);
                if (kRht) h ^= ((a.rht_signs >> (srow & 15)) & 1u) * 0x80008000u;
                sct[buf][srow][blk ^ (2 * ((srow >> 4) & 3))] = h;
            }
            if (kKind == 3 && tid < kTR) sdr[buf][tid] = sdreg;
        }
        const int next = tile + gridDim.x;
        if (next < n_tiles) {
            issue(next, buf ^ 1, sreg, sdreg);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const int tr = tile / tiles_c, tc = tile - tr * tiles_c;
        const int64_t r0 = (int64_t)tr * kTR, c0 = (int64_t)tc * kTC;
        const int64_t orow = c0 + 2 * p, ocol = r0 + 32 * (grp >> 1);
        const bool valid = orow < a.cols && ocol < a.rows;     // the same for both halves of a block
        if (kKind == 0) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(&stage[buf][0]) + (16 * grp) * 64 + (p ^ (8 * grp));
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                w[k] = src[k * 64];
                if (kRht) w[k] ^= ((a.rht_signs >> k) & 1u) * 0x80008000u;
            }
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const uint32_t sh = half ? 0u : 16u;     // even column: low bf16, odd: high
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = __uint_as_float((w[k] << sh) & 0xFFFF0000u);
                const int64_t oidx = (orow + half) * a.rows + ocol + 16 * hb;
                mx_encode_half<kRht, kSR>(v, valid, a.seed, a.tag, (uint64_t)oidx, a.out_e4m3 + oidx,
                                          hb ? nullptr : a.out_e8m0 + (oidx >> 5));
            }
            if (kDual) {
                // rowwise: thread (row, blk) encodes input row `row`'s 32 values of block blk of
                // this tile; its four 16-byte reads start at chunk rot = 2 (row & 1) + blk / 2, so
                // that each quarter-warp (two rows x four blocks) reads 8 distinct bank groups
                const int row = tid >> 2, blk = tid & 3, g = (row >> 4) & 3;
                const int rot = 2 * (row & 1) + (blk >> 1);
                const uint32_t* rw = reinterpret_cast<const uint32_t*>(&stage[buf][0]) + row * 64;
                uint4 w[4];   // w[qq] = chunk (qq + rot) & 3 of the block
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    w[qq] = *reinterpret_cast<const uint4*>(rw + 4 * ((4 * blk + ((qq + rot) & 3)) ^ (2 * g)));
                // undo the rotation with two conditional rotations (selects, no dynamic register
                // indexing): by 2, then by 1
                const bool r2 = (rot & 2) != 0, r1 = (rot & 1) != 0;
                uint4 u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 a0 = w[i], a2 = w[(i + 2) & 3];
                    u[i] = make_uint4(r2 ? a2.x : a0.x, r2 ? a2.y : a0.y, r2 ? a2.z : a0.z, r2 ? a2.w : a0.w);
                }
                float v[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 b0 = u[q], b1 = u[(q + 3) & 3];
                    const uint4 c = make_uint4(r1 ? b1.x : b0.x, r1 ? b1.y : b0.y, r1 ? b1.z : b0.z, r1 ? b1.w : b0.w);
                    bf16x2_to_f32(c.x, v + 8 * q);
                    bf16x2_to_f32(c.y, v + 8 * q + 2);
                    bf16x2_to_f32(c.z, v + 8 * q + 4);
                    bf16x2_to_f32(c.w, v + 8 * q + 6);
                }
                const int64_t r = r0 + row, c = c0 + 32 * blk;
                if (r < a.rows && c < a.cols)
                    mx_encode_block<false, kSR>(v, a.seed, a.tag2, (uint64_t)(r * a.cols + c),
                                                a.out2_e4m3 + r * a.cols + c, a.out2_e8m0 + (r * a.cols + c) / 32);
            }
        } else {
            const uint8_t* src = &stage[buf][0] + (16 * grp) * 64 + (p ^ (16 * grp));
            const uint32_t* sc = &sct[buf][16 * grp][(p >> 3) ^ (2 * grp)];
            uint32_t h[16];
            float sd[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                h[k] = e2m1x2_to_f16x2(src[k * 64]);
                asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[k]) : "r"(sc[k * 8]));
                sd[k] = kKind == 3 ? sdr[buf][16 * grp + k] : s_dec;
            }
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const uint32_t sel = half ? 0x3232u : 0x1010u;   // the column's f16 in both halves
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float f;
                    asm("{.reg .f16 l, u; mov.b32 {l, u}, %1; cvt.f32.f16 %0, l;}"
                        : "=f"(f) : "r"(__byte_perm(h[k], 0u, sel)));
                    v[k] = __fmul_rn(f, sd[k]);
                }
                const int64_t oidx = (orow + half) * a.rows + ocol + 16 * hb;
                mx_encode_half<kRht, kSR>(v, valid, a.seed, a.tag, (uint64_t)oidx, a.out_e4m3 + oidx,
                                          hb ? nullptr : a.out_e8m0 + (oidx >> 5));
            }
        }
        __syncthreads();
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
    if constexpr (kKind == 0) {
        if (a.transpose && a.out2_e4m3) {   // bf16: transposed + rowwise from one read
            const int64_t tiles_c = (a.cols + kTC - 1) / kTC, tiles_r = (a.rows + kTR - 1) / kTR;
            const int64_t n_tiles = tiles_c * tiles_r;
            static int per_sm[2][2] = {};
            int& occ = per_sm[kRht ? 1 : 0][kSR ? 1 : 0];
            if (occ <= 0) {
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, requant_t_kernel<0, kRht, kSR, true>,
                                                                  kTThreads, 0) != cudaSuccess || occ < 1) {
                    (void)cudaGetLastError();
                    occ = 4;
                }
            }
            int64_t g = (int64_t)num_sms() * occ;
            if (g > n_tiles) g = n_tiles;
            requant_t_kernel<0, kRht, kSR, true><<<(unsigned)g, kTThreads, 0, st>>>(a, (int)tiles_c, (int)n_tiles);
            return;
        }
    }
    if (a.transpose) {
        const int64_t tiles_c = (a.cols + kTC - 1) / kTC, tiles_r = (a.rows + kTR - 1) / kTR;
        const int64_t n_tiles = tiles_c * tiles_r;
        static int per_sm[4][2][2] = {};
        int& occ = per_sm[kKind][kRht ? 1 : 0][kSR ? 1 : 0];
        if (occ <= 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, requant_t_kernel<kKind, kRht, kSR>, kTThreads, 0) !=
                    cudaSuccess || occ < 1) {
                (void)cudaGetLastError();
                occ = 4;
            }
        }
        int64_t g = (int64_t)num_sms() * occ;
        if (g > n_tiles) g = n_tiles;
        requant_t_kernel<kKind, kRht, kSR><<<(unsigned)g, kTThreads, 0, st>>>(a, (int)tiles_c, (int)n_tiles);
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
        case 2: launch_requant_k<2>(a, st); break;
        default: launch_requant_k<3>(a, st); break;
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
