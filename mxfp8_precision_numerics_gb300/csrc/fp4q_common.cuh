// fp4q_common.cuh — device-side building blocks of the NVFP4 / MXFP8 kernels (sm_103a).
//
// Number formats (4bit.vizuara.ai §3-6; "Pretraining Large Language Models with NVFP4",
// "NVFP4 Format and Quantization Procedure"):
//   E2M1  s|ee|m, bias 1, exponent 0 subnormal: magnitudes {0,.5,1,1.5,2,3,4,6}
//   E4M3  s|eeee|mmm, bias 7, max 448 (0x7E), min subnormal 2^-9; 0x7F is NaN (never made)
//   E8M0  2^(byte - 127)
// Every fp32 operation of the quantization arithmetic goes through an explicit
// round-to-nearest intrinsic so that no multiply-add is contracted and each result is
// the single correctly rounded IEEE value the method's formulas name.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fp4q {

__device__ __forceinline__ float bf16_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// ---------------------------------------------------------------------------------------
// E4M3, round to nearest even with saturation to 448. Input any finite fp32.
//   normal range (|v| >= 2^-6): keep 3 of the 23 mantissa bits with a nearest-even carry
//   on the fp32 bit pattern (the carry may ripple into the exponent, which is exact);
//   subnormal range: the value in units of 2^-9 is rounded to the nearest even integer.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3_rne_sat(float v) {
    uint32_t u = __float_as_uint(v);
    uint32_t s = (u >> 24) & 0x80u;
    uint32_t a = u & 0x7FFFFFFFu;
    uint32_t c;
    if (a >= 0x43E00000u) {                       // |v| >= 448
        c = 0x7Eu;
    } else if (a >= 0x3C800000u) {                // |v| >= 2^-6: normal E4M3
        uint32_t r = a + 0x7FFFFu + ((a >> 20) & 1u);
        c = (r >> 20) - (120u << 3);              // rebias exponent 127 -> 7
    } else {
        float q = __fmul_rn(__uint_as_float(a), 512.0f);   // exact: power-of-two scale
        c = (uint32_t)__float2int_rn(q);          // nearest even in [0, 8]
    }
    return s | c;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float mag = (e == 0) ? __fmul_rn((float)m, 0.001953125f)          // m * 2^-9
                         : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (c & 0x80u) ? -mag : mag;
}

// E2M1 magnitude of a 4-bit code (sign in bit 3).
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    // bit pattern table of the eight magnitudes, four bits of fp32 exponent/mantissa each
    // is not needed: decode arithmetically.
    uint32_t e = (c >> 1) & 3u, m = c & 1u;
    float mag = (e == 0) ? (m ? 0.5f : 0.0f) : __uint_as_float(((e + 126u) << 23) | (m << 22));
    return (c & 8u) ? -mag : mag;
}

// ---------------------------------------------------------------------------------------
// E2M1, round to nearest with ties to the even code, saturating at 6; the sign is kept
// even when the magnitude rounds to zero. Decision thresholds are the midpoints between
// neighbouring grid values; at an exact midpoint the even code wins.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1_rne_alu(float v) {
    float a = fabsf(v);
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f)
               + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return c | ((__float_as_uint(v) >> 28) & 8u);
}

// Hardware conversion of two fp32 values to two E2M1 codes (round to nearest, satfinite).
// Used only where a device test has shown it equal to e2m1_rne_alu on every tie.
__device__ __forceinline__ uint32_t e2m1x2_cvt_rn(float lo, float hi) {
    uint32_t d;
    asm("{.reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %2, %1; cvt.u32.u8 %0, t;}"
        : "=r"(d) : "f"(lo), "f"(hi));
    return d;   // low nibble = lo, high nibble = hi
}

// ---------------------------------------------------------------------------------------
// MXFP8 block exponent, ceiling rule: the smallest integer e with amax <= 448 * 2^e,
// clamped to [-127, 127] ("FP4 Training on Blackwell", "The scaling math, worked").
// 448 = 1.75 * 2^8, so for amax = m * 2^E (m in [1,2)): e = E - 8 + (m > 1.75).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int mx_exponent(float amax) {
    uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (u < 0x00800000u) return -127;             // zero or subnormal: far below 448*2^-127
    if (u >= 0x7F800000u) return 127;             // infinite: no e fits, the clamp
    int E = (int)(u >> 23) - 127;
    int e = E - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^k as fp32 for k in [-149, 127] (k < -126: subnormal powers of two).
__device__ __forceinline__ float exp2i_wide(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}
// 2^k as fp32 for k in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2i(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// ---------------------------------------------------------------------------------------
// E4M3 stochastic rounding of t (|t| <= 448): floor(t/step + U) on the local grid with
// U = r16 / 2^16. Normal range: the 20 discarded mantissa bits F plus r16 << 4 carry into
// the kept bits exactly when F/2^20 + U >= 1. Subnormal range: in units of 2^-9 the value
// is m + f (m integer, f exact), rounded up when f >= 1 - U.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3_sr(float t, uint32_t r16) {
    uint32_t u = __float_as_uint(t);
    uint32_t s = (u >> 24) & 0x80u;
    uint32_t a = u & 0x7FFFFFFFu;
    uint32_t c;
    if (a >= 0x43E00000u) {
        c = 0x7Eu;
    } else if (a >= 0x3C800000u) {
        c = ((a + (r16 << 4)) >> 20) - (120u << 3);
    } else {
        float q = __fmul_rn(__uint_as_float(a), 512.0f);
        float m = truncf(q);
        float f = __fsub_rn(q, m);
        float thr = __fmul_rn((float)(65536u - r16), 1.52587890625e-05f);   // (2^16 - r) / 2^16
        c = (uint32_t)m + (f >= thr ? 1u : 0u);
    }
    return s | c;
}

// ---------------------------------------------------------------------------------------
// The same stochastic rounding done by the conversion unit, two values per instruction.
// cvt.rs.satfinite.e4m3x4.f32 packs four results; the result in byte 0 (fourth source
// operand) is rounded up exactly when F + (rbits[15:0] << 4) carries, the one in byte 2
// (second operand) likewise with rbits[31:16] -- the rule of e4m3_sr with r16 taken from
// those halves, including the subnormal range and saturation to 448. Bytes 1 and 3 draw on
// the same halves bit-reversed, so they would not be independent draws: they are fed zero.
// A device test checks this against the oracle's rounding on every grid point, midpoint
// and a million random (value, bits) pairs.
// Returns byte 0 = even, byte 2 = odd (bytes 1, 3 zero).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_sr_hw(float even, float odd, uint32_t rbits) {
    uint32_t d;
    asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %1, %3}, %4;"
        : "=r"(d) : "f"(0.0f), "f"(odd), "f"(even), "r"(rbits));
    return d;
}

// Four E4M3 codes, round to nearest even with saturation, byte k = code of the k-th
// argument (hardware conversion; first operand of each x2 instruction -> high byte).
__device__ __forceinline__ uint32_t e4m3x4_rn_hw(float a, float b, float c, float e) {
    uint32_t d;
    asm("{.reg .b16 l, h;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
        "mov.b32 %0, {l, h};}"
        : "=r"(d) : "f"(a), "f"(b), "f"(c), "f"(e));
    return d;
}

// Two packed E2M1 codes (low nibble = first value) -> f16x2 (low half = first value).
// Every E2M1 value is exact in f16.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t h;
    asm("{.reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(h) : "r"(byte));
    return h;
}

// Eight packed E2M1 codes times one E4M3 block scale times the fp32 tensor scale:
// out[j] = (E2M1(code_j) * scale) * s_dec. The first product is formed in f16x2 and is
// exact there (at most 2 x 4 significant bits, magnitudes in [2^-10, 2688]), so the only
// rounding is the fp32 multiply by s_dec, as in the definition.
// sc2 = the block scale as f16 in both halves.
__device__ __forceinline__ void dequant8_f16(uint32_t word, uint32_t sc2, float s_dec, float* out) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t h = e2m1x2_to_f16x2(word >> (8 * b));
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(sc2));
        float lo, hi;
        asm("{.reg .f16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h;}"
            : "=f"(lo), "=f"(hi) : "r"(h));
        out[2 * b] = __fmul_rn(lo, s_dec);
        out[2 * b + 1] = __fmul_rn(hi, s_dec);
    }
}

// An E4M3 scale byte as f16 in both halves of a word (exact: E4M3 values are f16 values).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t c) {
    uint32_t h;
    asm("{.reg .f16 s; cvt.rn.f16.f32 s, %1; mov.b32 %0, {s, s};}" : "=r"(h) : "f"(e4m3_to_f32(c)));
    return h;
}

// Sign flips of the random Hadamard transform applied to packed inputs: negation is exact,
// so flipping the source is the same as flipping the dequantized value.
// Nibble mask for eight E2M1 codes at transform positions p0 .. p0+7.
__device__ __forceinline__ uint32_t e2m1_sign_mask8(uint32_t signs, int p0) {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m |= ((signs >> (p0 + j)) & 1u) << (4 * j + 3);
    return m;
}
// Mask for two bf16 values (one 32-bit word) at transform positions p, p+1.
__device__ __forceinline__ uint32_t bf16_sign_mask2(uint32_t signs, int p) {
    return (((signs >> p) & 1u) << 15) | (((signs >> (p + 1)) & 1u) << 31);
}

// ---------------------------------------------------------------------------------------
// cp.async (16 bytes, zero-filled when !valid) into shared memory, its commit and wait.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kN>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kN) : "memory"); }

// ---------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of two 32x32->64 multiplies with the Weyl key schedule. Each product
// is one mul.wide.u32 (its low and high words are the round's lo and hi).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint64_t p0, p1;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
        const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
        const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// The eight 16-bit random slices for output elements [8*blk, 8*blk + 8) of tensor `tag`.
__device__ __forceinline__ uint4 sr_block8(uint64_t seed, uint32_t tag, uint64_t blk) {
    return philox4x32_10(make_uint4((uint32_t)blk, (uint32_t)(blk >> 32), tag, 0u),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t slice16(uint4 w, int j) {
    uint32_t x = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
    return (j & 1) ? (x >> 16) : (x & 0xFFFFu);
}

// ---------------------------------------------------------------------------------------
// Packed pairs of fp32 for add/sub/mul/fma.rn.f32x2 (sm_100+): each lane of a packed op
// rounds exactly like the scalar op; one instruction does two.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t d, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ---------------------------------------------------------------------------------------
// 16-point random Hadamard transform of v[0..15] in place: signs, butterflies at
// distances 1, 2, 4, 8 (Sylvester H16 = H2 (x) H8), then the exact scaling by 1/4.
// ("Pretraining Large Language Models with NVFP4", "Random Hadamard Transforms".)
// ---------------------------------------------------------------------------------------
// fwht16 is the butterflies alone (no signs, no 1/4); fwht16_quarter adds the 1/4. fwht16
// runs distance 1 on scalars and distances 2, 4, 8 on packed pairs (v[2m], v[2m+1]).
__device__ __forceinline__ void fwht16(float* v) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = __fadd_rn(a, b);
        v[i + 1] = __fsub_rn(a, b);
    }
    uint64_t p[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) p[m] = f32x2_pack(v[2 * m], v[2 * m + 1]);
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            if ((m & h) == 0) {
                const uint64_t s = f32x2_add(p[m], p[m + h]), d = f32x2_sub(p[m], p[m + h]);
                p[m] = s;
                p[m + h] = d;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) f32x2_unpack(p[m], v[2 * m], v[2 * m + 1]);
}

// t[j] = v[j] * s for 8 values, as 4 packed multiplies
__device__ __forceinline__ void mul8_f32x2(const float* v, float s, float* t) {
    const uint64_t s2 = f32x2_pack(s, s);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        f32x2_unpack(f32x2_mul(f32x2_pack(v[2 * m], v[2 * m + 1]), s2), t[2 * m], t[2 * m + 1]);
    }
}
__device__ __forceinline__ void fwht16_quarter(float* v) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = __fadd_rn(a, b);
                v[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

__device__ __forceinline__ void rht16_inplace(float* v, uint32_t signs) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if ((signs >> i) & 1u) v[i] = -v[i];
    fwht16_quarter(v);
}

// ---------------------------------------------------------------------------------------
// The combine wire format (4bit.vizuara.ai §11; "End-to-End 4-Bit Training" (Thinking
// Machines), 合并阶段): rotate groups of 32 values (sign flips, Sylvester H32 butterflies at
// distances 1, 2, 4, 8, 16 in fp32, then one multiply by RN(1/sqrt 32)), then S2F6 (a signed
// 8-bit integer over 64) with one E8M0 scale per 32: e = the smallest integer with
// amax <= (127/64) 2^e, clamped to [-127, 127]; q = round-half-even(y 2^(6-e)) in [-128, 127].
// ---------------------------------------------------------------------------------------
constexpr float kRht32Scale = 0.17677669529663688f;   // RN(1/sqrt(32)) = 0x3E3504F3

// Butterflies at distance 1 on scalars; distances 2..16 on packed pairs (v[2m], v[2m+1]) with
// add/sub.rn.f32x2 (each lane of a packed op rounds like the scalar op); then a packed
// multiply by `scale`. Results are those of the scalar stages in the same order.
__device__ __forceinline__ void fwht32_scaled(float (&v)[32], float scale) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = __fadd_rn(a, b);
        v[i + 1] = __fsub_rn(a, b);
    }
    uint64_t p[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) p[m] = f32x2_pack(v[2 * m], v[2 * m + 1]);
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            if ((m & h) == 0) {
                const uint64_t s = f32x2_add(p[m], p[m + h]), d = f32x2_sub(p[m], p[m + h]);
                p[m] = s;
                p[m + h] = d;
            }
        }
    }
    const uint64_t sc2 = f32x2_pack(scale, scale);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        f32x2_unpack(f32x2_mul(p[m], sc2), v[2 * m], v[2 * m + 1]);
    }
}

// forward: signs, butterflies, scale
__device__ __forceinline__ void rht32_forward(float (&v)[32], uint32_t signs) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ (((signs >> i) & 1u) << 31));
    fwht32_scaled(v, kRht32Scale);
}

// inverse: butterflies, scale, signs
__device__ __forceinline__ void rht32_inverse(float (&v)[32], uint32_t signs) {
    fwht32_scaled(v, kRht32Scale);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ (((signs >> i) & 1u) << 31));
}

// S2F6 block exponent (ceiling rule with the format's maximum 127/64 = 1.111111b):
// amax = m 2^E, m in [1, 2): e = E + (m > 127/64); subnormal amax: -127 up to 127 * 2^-133.
__device__ __forceinline__ int s2f6_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (u < 0x00800000u) return u <= 0x007F0000u ? -127 : -126;
    const int e = (int)(u >> 23) - 127 + ((u & 0x7FFFFFu) > 0x7E0000u ? 1 : 0);
    return e > 127 ? 127 : e;
}

// 32 rotated values -> 32 S2F6 bytes (out, 8 words) and the E8M0 byte.
__device__ __forceinline__ uint32_t s2f6_encode32(const float (&y)[32], uint32_t (&out)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(y[i]));
    const int e = s2f6_exponent(amax);
    const float inv = exp2i(-e);        // y 2^-e, then x 64: both exact (a value that is
                                        // subnormal after the first step is < 2^-120 and rounds to 0)
    // Clamp to [-128, 127], then round half to even by adding 1.5 * 2^23: in [2^23, 2^24) the
    // spacing is 1, so the sum is 1.5 * 2^23 + RNE(t) and its low byte is RNE(t) in two's
    // complement (clamping first or last gives the same code). No integer conversion is needed.
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float t = __fmul_rn(__fmul_rn(y[4 * w + j], inv), 64.0f);
            b[j] = __float_as_uint(__fadd_rn(fminf(fmaxf(t, -128.0f), 127.0f), 12582912.0f));
        }
        out[w] = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
    }
    return (uint32_t)(e + 127);
}

// one S2F6 word (4 codes) with E8M0 byte sc -> 4 exact fp32 values. Code c (int8) is taken
// as the float 2^23 + (c + 128) (its biased byte under the exponent bits of 2^23), less
// 2^23 + 128 (exact), times the power-of-two step (exact).
__device__ __forceinline__ void s2f6_decode4(uint32_t word, uint32_t sc, float* out) {
    const float step = exp2i_wide((int)sc - 127 - 6);
    const uint32_t biased = word ^ 0x80808080u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float f = __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7440u + j));
        out[j] = __fmul_rn(__fsub_rn(f, 8388736.0f), step);
    }
}

}  // namespace fp4q
