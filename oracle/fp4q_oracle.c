/*
 * fp4q_oracle.c — plain, slow CPU oracle for the NVFP4 / MXFP8 arithmetic of the
 * 4-bit linear layer (forward NVFP4, backward MXFP8 with stochastic rounding and a
 * 16-point random Hadamard transform).
 *
 * TEST INFRASTRUCTURE ONLY. This library exists so that the CUDA library can be
 * checked against an independent statement of the method. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no code,
 * header, table or constant generator with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (web pages, cited by title and section):
 *   [VZ]  "End-to-End 4-Bit Training", rebuilt on one B200 (4bit.vizuara.ai):
 *         §3-4 (E2M1 table, E4M3), §5-6 (block scale, outer scale, round_float),
 *         §7-10 (GEMM, transposes, stochastic rounding, requantization), §11 (RHT).
 *   [NV]  "Pretraining Large Language Models with NVFP4" (arXiv 2509.25149) summary:
 *         "NVFP4 Format and Quantization Procedure" steps 1-5, "Random Hadamard
 *         Transforms", "Two-Dimensional Weight Scaling", "Stochastic Rounding".
 *   [TML] "End-to-End 4-Bit Training" (Thinking Machines; Chinese rendering):
 *         "Blackwell 架构上的低精度格式" (E4M3 96 = 0|1101|100, -54 -> -6 with scale 9),
 *         "基于随机舍入的重量化" (5.4 -> 4.5, re-quantize with SR).
 *   [AC]  "FP4 Training on Blackwell" (aicassindra.com): "The E2M1 format",
 *         "The scaling math, worked" (power-of-two ceiling scale), "Stochastic
 *         rounding", "Hadamard rotations".
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *         1, 2, 3", SC'11, section 4 (Philox round function and key schedule).
 *
 * Readings where the pages are silent or disagree:
 *   - E2M1 ties go to the even code (round-to-nearest-even, [NV] step 4); a value
 *     that rounds to zero keeps its sign ([VZ] §6 round_float uses copysign).
 *   - The scale arithmetic follows [NV] steps 1-4 literally in fp32:
 *       s_enc = 2688 / amax ; s_dec = 1 / s_enc ;
 *       sb = e4m3_rne((amax_b / 6) * s_enc) ; s_enc_b = 1 / (fp32(sb) * s_dec) ;
 *       code = e2m1_rne(x * s_enc_b).
 *     amax == 0 or a non-finite s_enc gives s_enc = s_dec = 1. A block scale that
 *     rounds to E4M3 zero is raised to the smallest code 0x01 ([VZ] §13 kernel).
 *   - MXFP8 block exponent: the smallest e with amax <= 448 * 2^e (ceiling rule of
 *     [AC] "The scaling math, worked" and [VZ] §6 "nearest usable power of two would
 *     be 16"), clamped to [-127, 127]; E8M0 byte = e + 127.
 *   - Stochastic rounding is floor(t + U) in units of the local grid step ([VZ] §6
 *     round_float, mode "sr"), with U = R16 / 65536 and R16 a 16-bit slice of a
 *     Philox4x32-10 output (see sr_bits16 below for the exact counter layout).
 *   - RHT16: y = (1/4) * H16 * (s o x) along the contiguous dimension, Sylvester
 *     H16 = H2 (x) H8 evaluated as a fast Walsh-Hadamard transform in fp32 with
 *     butterfly distances 1, 2, 4, 8 (the order the Kronecker recursion implies),
 *     then multiplied by 0.25 (exact).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * All fp32 arithmetic below is single IEEE operations with round-to-nearest-even and
 * no contraction; encodings are searched in double, where every step is exact.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* bit casts                                                                  */
/* ------------------------------------------------------------------------- */
static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bf16_value(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* ------------------------------------------------------------------------- */
/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is subnormal.  */
/* [VZ] §3-4 table; [AC] "The E2M1 format".                                   */
/* ------------------------------------------------------------------------- */
EXPORT double orc_e2m1_decode(uint32_t code)
{
    uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m                      /* {0, 0.5}      */
                          : ldexp(1.0 + 0.5 * (double)m, (int)e - 1); /* 2^(e-1)(1+m/2) */
    return s ? -mag : mag;
}

/* Round to the nearest E2M1 value, ties to the even code, saturating at 6.
 * Plain nearest search over the eight magnitudes. */
EXPORT uint32_t orc_e2m1_encode_rne(float v)
{
    double a = fabs((double)v);
    uint32_t best = 7;                       /* |v| >= 6 saturates to 6 */
    if (a < 6.0) {
        double best_d = INFINITY;
        for (uint32_t c = 0; c < 8; ++c) {
            double d = fabs(a - orc_e2m1_decode(c));
            if (d < best_d || (d == best_d && (c & 1u) == 0)) { best = c; best_d = d; }
        }
    }
    uint32_t sign = (bits_from_f32(v) >> 31) & 1u;
    return (sign << 3) | best;
}

/* Stochastic E2M1 rounding, floor(t + U) on the E2M1 grid ([VZ] §9 worked example
 * 2.25 -> 2 or 3). Used only by the oracle's own statistical pins. */
EXPORT uint32_t orc_e2m1_encode_sr(float v, uint32_t r16)
{
    double a = fabs((double)v);
    uint32_t sign = (bits_from_f32(v) >> 31) & 1u;
    if (a >= 6.0) return (sign << 3) | 7u;
    uint32_t lo = 0;
    for (uint32_t c = 0; c < 8; ++c) if (orc_e2m1_decode(c) <= a) lo = c;
    double va = orc_e2m1_decode(lo), vb = orc_e2m1_decode(lo + 1);
    double frac = (a - va) / (vb - va);
    double u = (double)r16 / 65536.0;
    uint32_t c = (frac >= 1.0 - u) ? lo + 1 : lo;
    return (sign << 3) | c;
}

/* ------------------------------------------------------------------------- */
/* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448, min 2^-9.     */
/* [VZ] §4; [TML] "Blackwell 架构上的低精度格式" (96 = 0|1101|100).            */
/* 0x7F / 0xFF are NaN and are never produced here.                           */
/* ------------------------------------------------------------------------- */
EXPORT double orc_e4m3_decode(uint32_t code)
{
    uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6)
                          : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* largest magnitude code c in [0, 0x7E] with decode(c) <= a  (a >= 0, a < 448) */
static uint32_t e4m3_floor_code(double a)
{
    uint32_t lo = 0, hi = 0x7E;            /* decode is increasing in the code */
    while (lo < hi) {
        uint32_t mid = (lo + hi + 1) / 2;
        if (orc_e4m3_decode(mid) <= a) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* Round to the nearest E4M3 value, ties to the even code, saturating to 448. */
EXPORT uint32_t orc_e4m3_encode_rne_sat(float v)
{
    double a = fabs((double)v);
    uint32_t sign = (bits_from_f32(v) >> 31) & 1u;
    uint32_t c;
    if (a >= 448.0) {
        c = 0x7E;
    } else {
        uint32_t lo = e4m3_floor_code(a);
        double dl = a - orc_e4m3_decode(lo);
        double dh = orc_e4m3_decode(lo + 1) - a;
        if (dl < dh) c = lo;
        else if (dh < dl) c = lo + 1;
        else c = (lo & 1u) ? lo + 1 : lo;
    }
    return (sign << 7) | c;
}

/* Stochastic E4M3 rounding: q = floor(t/step + U) * step on the local grid step,
 * U = r16 / 2^16. Grid points are fixed points. |t| must not exceed 448 (the MXFP8
 * ceiling exponent guarantees it); larger inputs saturate. */
EXPORT uint32_t orc_e4m3_encode_sr(float v, uint32_t r16)
{
    double a = fabs((double)v);
    uint32_t sign = (bits_from_f32(v) >> 31) & 1u;
    uint32_t c;
    if (a >= 448.0) {
        c = 0x7E;
    } else {
        uint32_t lo = e4m3_floor_code(a);
        double va = orc_e4m3_decode(lo), vb = orc_e4m3_decode(lo + 1);
        double frac = (a - va) / (vb - va);          /* exact: vb - va is 2^k   */
        double u = (double)r16 / 65536.0;
        c = (frac >= 1.0 - u) ? lo + 1 : lo;         /* floor(frac + u) == 1    */
    }
    return (sign << 7) | c;
}

/* ------------------------------------------------------------------------- */
/* E8M0 / power-of-two block exponent, ceiling rule:                          */
/* the smallest integer e with amax <= vmax * 2^e, clamped to [-127, 127].     */
/* [AC] "The scaling math, worked": scale = 2^ceil(log2(amax / vmax)).         */
/* ------------------------------------------------------------------------- */
EXPORT int orc_pow2_ceil_exponent(double amax, double vmax)
{
    int e = -127;
    while (e < 127 && amax > vmax * ldexp(1.0, e)) ++e;
    return e;
}

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon et al., SC'11 §4).                                   */
/* ------------------------------------------------------------------------- */
EXPORT void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B9u;   /* Weyl key schedule */
        k1 += 0xBB67AE85u;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The 16 random bits that stochastic rounding spends on output element `idx`
 * (its linear index in the row-major OUTPUT layout) of the tensor tagged `tag`:
 * Philox4x32-10 with key (seed lo, seed hi) and counter (idx>>3 lo, idx>>3 hi, tag, 0)
 * yields four 32-bit words = eight 16-bit slices; element idx takes word (idx>>1)&3,
 * low half if idx is even, high half if odd. */
EXPORT uint32_t orc_sr_bits16(uint64_t seed, uint32_t tag, uint64_t idx)
{
    uint64_t blk = idx >> 3;
    uint32_t ctr[4] = { (uint32_t)blk, (uint32_t)(blk >> 32), tag, 0u };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t w = out[(idx >> 1) & 3u];
    return (idx & 1u) ? (w >> 16) : (w & 0xFFFFu);
}

/* ------------------------------------------------------------------------- */
/* Per-tensor amax and the global scales ([NV] step 1).                       */
/* ------------------------------------------------------------------------- */
EXPORT float orc_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld)
{
    float m = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(bf16_value(x[r * ld + c]));
            if (a > m) m = a;
        }
    return m;
}

/* s_enc = (6 * 448) / amax, s_dec = 1 / s_enc, both fp32. */
EXPORT void orc_global_scales(float amax, float* s_enc_out, float* s_dec_out)
{
    float s_enc = 2688.0f / amax;
    if (!(amax > 0.0f) || !isfinite(s_enc)) s_enc = 1.0f;
    *s_enc_out = s_enc;
    *s_dec_out = 1.0f / s_enc;
}

/* One NVFP4 block scale from the block amax ([NV] steps 2-3): returns the E4M3
 * code of (amax_b / 6) * s_enc, raised to 0x01 if it rounds to zero. */
EXPORT uint32_t orc_block_scale_code(float amax_b, float s_enc)
{
    float s_dec_b = amax_b / 6.0f;
    float v = s_dec_b * s_enc;
    uint32_t sb = orc_e4m3_encode_rne_sat(v) & 0x7Fu;
    if (sb == 0) sb = 1;
    return sb;
}

/* The local encode scale s_enc_b = 1 / (fp32(sb) * s_dec) ([NV] step 3). */
EXPORT float orc_block_encode_scale(uint32_t sb, float s_dec)
{
    float dsb = (float)orc_e4m3_decode(sb);
    float p = dsb * s_dec;
    return 1.0f / p;
}

static void put_code(uint8_t* codes, int64_t row_bytes, int64_t r, int64_t c, uint32_t code)
{
    uint8_t* b = &codes[r * row_bytes + (c >> 1)];
    if (c & 1) *b = (uint8_t)((*b & 0x0Fu) | (code << 4));
    else       *b = (uint8_t)((*b & 0xF0u) | (code & 0x0Fu));
}

static uint32_t get_code(const uint8_t* codes, int64_t row_bytes, int64_t r, int64_t c)
{
    uint8_t b = codes[r * row_bytes + (c >> 1)];
    return (c & 1) ? (uint32_t)(b >> 4) : (uint32_t)(b & 0x0Fu);
}

/* ------------------------------------------------------------------------- */
/* NVFP4 1D quantize: blocks of 16 contiguous values along each row.          */
/* [NV] "NVFP4 Format and Quantization Procedure" steps 1-4; [VZ] §6 nvfp4.   */
/* codes: [rows][cols/2], element 2j in the low nibble; scales: [rows][cols/16]. */
/* amax_in: if non-NULL, the per-tensor amax to use instead of computing it.  */
/* ------------------------------------------------------------------------- */
EXPORT void orc_quantize_1d(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            const float* amax_in, uint8_t* codes, uint8_t* scales,
                            float* amax_out, float* s_dec_out)
{
    float amax = amax_in ? *amax_in : orc_amax_bf16(x, rows, cols, ld);
    float s_enc, s_dec;
    orc_global_scales(amax, &s_enc, &s_dec);
    int64_t nb = cols / 16;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(bf16_value(x[r * ld + b * 16 + i]));
                if (a > amax_b) amax_b = a;
            }
            uint32_t sb = orc_block_scale_code(amax_b, s_enc);
            float s_enc_b = orc_block_encode_scale(sb, s_dec);
            scales[r * nb + b] = (uint8_t)sb;
            for (int i = 0; i < 16; ++i) {
                float v = bf16_value(x[r * ld + b * 16 + i]) * s_enc_b;
                put_code(codes, cols / 2, r, b * 16 + i, orc_e2m1_encode_rne(v));
            }
        }
    }
    if (amax_out) *amax_out = amax;
    *s_dec_out = s_dec;
}

/* ------------------------------------------------------------------------- */
/* NVFP4 1D quantize with a per-row (per-token) FP32 outer scale and, when     */
/* four_six is set, the Four Over Six choice of block scale.                   */
/* [VZ] §10: 4/6 tries a second scale per block that puts the block maximum   */
/* on 4 instead of 6 and keeps the version with the smaller error (the choice  */
/* lives in the block scale; activations only), and the activation outer      */
/* scale is computed separately for each token's row (QLinearFn listing:      */
/* outer="row", four_six=True for x; outer="tensor" for w). [TML] "方案细节":   */
/* 4/6 on activations, not weights; per-token outer scale for activations.    */
/* Readings where the pages are silent:                                       */
/*   - a row's s_enc / s_dec are orc_global_scales of that row's own amax;    */
/*   - candidate c (target c = 6 or c = 4) is the per-tensor block rule with  */
/*     6 replaced by c: sb_c = e4m3_rne_sat((amax_b / c) * s_enc), raised to  */
/*     0x01 if 0; s_enc_b = 1 / (fp32(sb_c) * s_dec); y_i = x_i * s_enc_b;    */
/*     code_i = e2m1_rne(y_i). Where (amax_b / 4) * s_enc exceeds 448 the      */
/*     scale saturates and the maximum lands between 4 and 6;                 */
/*   - "error" is the block's squared error. With S_c = fp32(sb_c) and q_i    */
/*     the E2M1 value of code_i, x_i - x^_i = s_dec * S_c * (y_i - q_i) up to */
/*     the rounding of y_i, and s_dec is the same for both candidates, so the */
/*     compared quantity is E_c = (sum_i (y_i - q_i)^2) * S_c^2 in fp32. Each */
/*     y_i - q_i is exact (q_i is the grid point nearest y_i, |y_i| < 12);    */
/*     the squares go into two sums, one over the even positions and one over */
/*     the odd, each built in index order with fused multiply-adds (one       */
/*     rounding per step); E_c = (even + odd) * S_c^2 (S_c^2 is exact);       */
/*   - the 4 candidate is kept only if E_4 < E_6 (a tie keeps 6).             */
/* ------------------------------------------------------------------------- */

/* One candidate for the 16 bf16 values xb (amax_b = max |xb|): its scale code,
 * its 16 codes and its error E_c. */
EXPORT void orc_nvfp4_block_candidate(const uint16_t* xb, float target, float s_enc, float s_dec,
                                      uint32_t* sb_out, uint8_t* codes16, float* err_out)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(bf16_value(xb[i]));
        if (a > amax_b) amax_b = a;
    }
    uint32_t sb = orc_e4m3_encode_rne_sat((amax_b / target) * s_enc) & 0x7Fu;
    if (sb == 0) sb = 1;
    float s_enc_b = orc_block_encode_scale(sb, s_dec);
    float even = 0.0f, odd = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float y = bf16_value(xb[i]) * s_enc_b;
        uint32_t code = orc_e2m1_encode_rne(y);
        float d = y - (float)orc_e2m1_decode(code);
        if (i & 1) odd = fmaf(d, d, odd);
        else       even = fmaf(d, d, even);
        codes16[i] = (uint8_t)code;
    }
    float S = (float)orc_e4m3_decode(sb);
    *sb_out = sb;
    *err_out = (even + odd) * (S * S);
}

/* codes [rows][cols/2], scales [rows][cols/16], s_dec_rows [rows]. */
EXPORT void orc_quantize_1d_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                 int four_six, uint8_t* codes, uint8_t* scales, float* s_dec_rows)
{
    int64_t nb = cols / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * ld;
        float s_enc, s_dec;
        orc_global_scales(orc_amax_bf16(xr, 1, cols, cols), &s_enc, &s_dec);
        for (int64_t b = 0; b < nb; ++b) {
            uint32_t sb, sb4;
            uint8_t c6[16], c4[16];
            float e6, e4;
            orc_nvfp4_block_candidate(xr + b * 16, 6.0f, s_enc, s_dec, &sb, c6, &e6);
            const uint8_t* c = c6;
            if (four_six) {
                orc_nvfp4_block_candidate(xr + b * 16, 4.0f, s_enc, s_dec, &sb4, c4, &e4);
                if (e4 < e6) { sb = sb4; c = c4; }
            }
            scales[r * nb + b] = (uint8_t)sb;
            for (int i = 0; i < 16; ++i) put_code(codes, cols / 2, r, b * 16 + i, c[i]);
        }
        s_dec_rows[r] = s_dec;
    }
}

/* ------------------------------------------------------------------------- */
/* NVFP4 2D quantize: one scale per 16x16 tile ([NV] "Two-Dimensional Weight   */
/* Scaling"; [VZ] §8). tile_scales: [rows/16][cols/16].                        */
/* ------------------------------------------------------------------------- */
EXPORT void orc_quantize_2d(const uint16_t* w, int64_t rows, int64_t cols, int64_t ld,
                            const float* amax_in, uint8_t* codes, uint8_t* tile_scales,
                            float* amax_out, float* s_dec_out)
{
    float amax = amax_in ? *amax_in : orc_amax_bf16(w, rows, cols, ld);
    float s_enc, s_dec;
    orc_global_scales(amax, &s_enc, &s_dec);
    int64_t tr = rows / 16, tc = cols / 16;
    for (int64_t ti = 0; ti < tr; ++ti) {
        for (int64_t tj = 0; tj < tc; ++tj) {
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float a = fabsf(bf16_value(w[(ti * 16 + i) * ld + tj * 16 + j]));
                    if (a > amax_b) amax_b = a;
                }
            uint32_t sb = orc_block_scale_code(amax_b, s_enc);
            float s_enc_b = orc_block_encode_scale(sb, s_dec);
            tile_scales[ti * tc + tj] = (uint8_t)sb;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float v = bf16_value(w[(ti * 16 + i) * ld + tj * 16 + j]) * s_enc_b;
                    put_code(codes, cols / 2, ti * 16 + i, tj * 16 + j, orc_e2m1_encode_rne(v));
                }
        }
    }
    if (amax_out) *amax_out = amax;
    *s_dec_out = s_dec;
}

/* ------------------------------------------------------------------------- */
/* NVFP4 dequantize ([VZ] §6: value = code x block scale x outer scale).       */
/* scale_kind 1: scales [rows][cols/16]; 2: tile scales [rows/16][cols/16].    */
/* out_f32: fp32 value (the exact product rounded once); out_f64: exact value. */
/* ------------------------------------------------------------------------- */
static double nvfp4_value(const uint8_t* codes, const uint8_t* scales, int scale_kind,
                          double s_dec, int64_t rows, int64_t cols, int64_t r, int64_t c)
{
    (void)rows;
    uint32_t sb = (scale_kind == 2) ? scales[(r / 16) * (cols / 16) + c / 16]
                                    : scales[r * (cols / 16) + c / 16];   /* kinds 1 and 3 */
    return orc_e2m1_decode(get_code(codes, cols / 2, r, c)) * orc_e4m3_decode(sb) * s_dec;
}

EXPORT void orc_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, int scale_kind,
                              float s_dec, int64_t rows, int64_t cols,
                              float* out_f32, double* out_f64)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            double v = nvfp4_value(codes, scales, scale_kind, (double)s_dec, rows, cols, r, c);
            if (out_f32) out_f32[r * cols + c] = (float)v;
            if (out_f64) out_f64[r * cols + c] = v;
        }
}

/* NVFP4 with 1D scales and a per-row outer scale (orc_quantize_1d_rows):
 * value = code x block scale x s_dec_rows[r]. */
EXPORT void orc_dequant_nvfp4_rows(const uint8_t* codes, const uint8_t* scales, const float* s_dec_rows,
                                   int64_t rows, int64_t cols, float* out_f32, double* out_f64)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            double v = nvfp4_value(codes, scales, 1, (double)s_dec_rows[r], rows, cols, r, c);
            if (out_f32) out_f32[r * cols + c] = (float)v;
            if (out_f64) out_f64[r * cols + c] = v;
        }
}

/* MXFP8 dequantize: value = e4m3 x 2^(e8m0 - 127); blocks of 32 along rows. */
EXPORT void orc_dequant_mxfp8(const uint8_t* e4m3, const uint8_t* e8m0, int64_t rows,
                              int64_t cols, double* out_f64)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out_f64[r * cols + c] = orc_e4m3_decode(e4m3[r * cols + c])
                                    * ldexp(1.0, (int)e8m0[r * (cols / 32) + c / 32] - 127);
}

/* ------------------------------------------------------------------------- */
/* 16-point random Hadamard transform on one group, in place, fp32:           */
/* signs first (bit i set -> negate element i), then the Walsh-Hadamard        */
/* butterflies at distances 1, 2, 4, 8, then x 1/4 (= 1/sqrt(16)).             */
/* [NV] "Random Hadamard Transforms"; [AC] "Hadamard rotations".               */
/* ------------------------------------------------------------------------- */
EXPORT void orc_rht16_group(float* v, uint32_t signs)
{
    for (int i = 0; i < 16; ++i)
        if ((signs >> i) & 1u) v[i] = -v[i];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int i = 0; i < 16; ++i) v[i] = v[i] * 0.25f;
}

/* rht16 on a [rows][cols] tensor (fp32 or bf16 input), along cols. */
EXPORT void orc_rht16(const void* in, int in_is_bf16, float* out, int64_t rows, int64_t cols,
                      uint32_t signs)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < cols / 16; ++g) {
            float v[16];
            for (int i = 0; i < 16; ++i) {
                int64_t k = r * cols + g * 16 + i;
                v[i] = in_is_bf16 ? bf16_value(((const uint16_t*)in)[k]) : ((const float*)in)[k];
            }
            orc_rht16_group(v, signs);
            for (int i = 0; i < 16; ++i) out[r * cols + g * 16 + i] = v[i];
        }
}

/* ------------------------------------------------------------------------- */
/* MXFP8 quantize of one block of 32 fp32 values ([VZ] §6 MXFP8; [AC] ceiling  */
/* scale with vmax = 448). rounding 0 = RNE, 1 = stochastic; out_idx0 is the   */
/* output linear index of v[0] (RNG counter).                                 */
/* ------------------------------------------------------------------------- */
EXPORT void orc_mxfp8_block(const float* v, int rounding, uint64_t seed, uint32_t tag,
                            uint64_t out_idx0, uint8_t* out_e4m3, uint8_t* out_e8m0)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
    int e = orc_pow2_ceil_exponent(amax, 448.0);
    *out_e8m0 = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) {
        float t = (float)ldexp((double)v[i], -e);       /* exact power-of-two scaling */
        out_e4m3[i] = (uint8_t)(rounding ? orc_e4m3_encode_sr(t, orc_sr_bits16(seed, tag, out_idx0 + (uint64_t)i))
                                         : orc_e4m3_encode_rne_sat(t));
    }
}

/* ------------------------------------------------------------------------- */
/* Dequantize -> [transpose] -> [RHT16] -> MXFP8 (SR or RNE).                  */
/* [VZ] §9-10 (dequantize, transpose, re-quantize to MXFP8 with SR);           */
/* [TML] "基于随机舍入的重量化"; [NV] "Random Hadamard Transforms" (wgrad only). */
/* in_kind: 0 = bf16 [rows][cols]; 1 = NVFP4 with 1D scales; 2 = NVFP4 with    */
/*          16x16 tile scales; 3 = NVFP4 with 1D scales and a per-row outer     */
/*          scale s_dec_rows[rows] (s_dec unused).                             */
/* Output: transpose ? [cols][rows] : [rows][cols], E8M0 per 32 along the       */
/*         output's contiguous dimension.                                      */
/* ------------------------------------------------------------------------- */
/* Output rows [orow_begin, orow_end) only; out_e4m3 / out_e8m0 hold just those rows. */
EXPORT void orc_requant_mxfp8_rows(int in_kind, const void* in, const uint8_t* in_scales, float s_dec,
                                   const float* s_dec_rows, int64_t rows, int64_t cols, int transpose, int rht, uint32_t rht_signs,
                                   int rounding, uint64_t seed, uint32_t tag,
                                   int64_t orow_begin, int64_t orow_end,
                                   uint8_t* out_e4m3, uint8_t* out_e8m0)
{
    int64_t ocols = transpose ? rows : cols;
    float v[32];
    for (int64_t orow = orow_begin; orow < orow_end; ++orow) {
        for (int64_t ob = 0; ob < ocols / 32; ++ob) {
            for (int i = 0; i < 32; ++i) {
                int64_t oc = ob * 32 + i;
                int64_t r = transpose ? oc : orow;     /* source coordinates */
                int64_t c = transpose ? orow : oc;
                if (in_kind == 0) v[i] = bf16_value(((const uint16_t*)in)[r * cols + c]);
                else v[i] = (float)nvfp4_value((const uint8_t*)in, in_scales, in_kind,
                                               in_kind == 3 ? (double)s_dec_rows[r] : (double)s_dec,
                                               rows, cols, r, c);
            }
            if (rht) { orc_rht16_group(v, rht_signs); orc_rht16_group(v + 16, rht_signs); }
            int64_t lr = orow - orow_begin;
            orc_mxfp8_block(v, rounding, seed, tag, (uint64_t)(orow * ocols + ob * 32),
                            &out_e4m3[lr * ocols + ob * 32], &out_e8m0[lr * (ocols / 32) + ob]);
        }
    }
}

EXPORT void orc_requant_mxfp8(int in_kind, const void* in, const uint8_t* in_scales, float s_dec,
                              const float* s_dec_rows, int64_t rows, int64_t cols, int transpose, int rht, uint32_t rht_signs,
                              int rounding, uint64_t seed, uint32_t tag,
                              uint8_t* out_e4m3, uint8_t* out_e8m0)
{
    orc_requant_mxfp8_rows(in_kind, in, in_scales, s_dec, s_dec_rows, rows, cols, transpose, rht, rht_signs,
                           rounding, seed, tag, 0, transpose ? cols : rows, out_e4m3, out_e8m0);
}

/* ------------------------------------------------------------------------- */
/* The MoE combine wire format: RHT32 + block-scaled S2F6.                    */
/* [VZ] §11: rotate 32 values at a time (flip signs by a fixed random         */
/* pattern, then 32 sums and differences of all of them, each divided by      */
/* sqrt(32)); quantize to S2F6, an 8-bit signed integer divided by 64         */
/* (-2 .. 127/64 in steps of 1/64), with one power-of-two scale per 32         */
/* values (8.25 bits per value); the receiver dequantizes and adds up the      */
/* arrivals, then undoes the rotation. [TML] "合并阶段": RHT32, then blocked    */
/* S2F6 with an E8M0 scale per 32; dequantize and aggregate on arrival, then  */
/* inverse Hadamard.                                                          */
/* Readings where the pages are silent:                                       */
/*   - the rotation is y = c * H32 (s o x) with c = RN(1/sqrt(32)) in fp32:   */
/*     signs first, butterflies at distances 1, 2, 4, 8, 16, then one         */
/*     multiply by c per value; its inverse applies the same butterflies and  */
/*     c, then the signs (H32 is symmetric and (H32/sqrt 32)^2 = I);          */
/*   - the block exponent is the ceiling rule of the MXFP8 path with the      */
/*     S2F6 maximum 127/64: the smallest e with amax <= (127/64) 2^e, clamped */
/*     to [-127, 127], E8M0 byte e + 127; nothing saturates below the clamp;  */
/*   - q = round-half-even(y * 2^(6 - e)), clamped to [-128, 127], stored as  */
/*     a two's-complement byte; value q * 2^(e - 6);                          */
/*   - arrivals are summed in fp32 in index order (slot 0 first), in the      */
/*     rotated domain, and the sum is rotated back once (the rotation is      */
/*     linear).                                                               */
/* ------------------------------------------------------------------------- */
static const float kRhtC32 = 0.17677669529663688f;   /* RN(1/sqrt(32)) */

static void fwht32(float* v)
{
    for (int h = 1; h < 32; h <<= 1)
        for (int i = 0; i < 32; ++i)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
}

/* Forward rotation of one group of 32, in place. */
EXPORT void orc_rht32_group(float* v, uint32_t signs)
{
    for (int i = 0; i < 32; ++i)
        if ((signs >> i) & 1u) v[i] = -v[i];
    fwht32(v);
    for (int i = 0; i < 32; ++i) v[i] = v[i] * kRhtC32;
}

/* Inverse rotation of one group of 32, in place. */
EXPORT void orc_irht32_group(float* v, uint32_t signs)
{
    fwht32(v);
    for (int i = 0; i < 32; ++i) v[i] = v[i] * kRhtC32;
    for (int i = 0; i < 32; ++i)
        if ((signs >> i) & 1u) v[i] = -v[i];
}

/* S2F6 block quantize of 32 fp32 values: codes (two's-complement bytes) and the
 * E8M0 byte. */
EXPORT void orc_s2f6_block(const float* y, uint8_t* codes, uint8_t* e8m0)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) if (fabs((double)y[i]) > amax) amax = fabs((double)y[i]);
    int e = orc_pow2_ceil_exponent(amax, 127.0 / 64.0);
    *e8m0 = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) {
        double t = ldexp((double)y[i], 6 - e);           /* exact */
        double q = nearbyint(t);                         /* ties to even (default mode) */
        if (q > 127.0) q = 127.0;
        if (q < -128.0) q = -128.0;
        codes[i] = (uint8_t)(int8_t)q;
    }
}

EXPORT double orc_s2f6_decode(uint8_t code, uint8_t e8m0)
{
    return ldexp((double)(int8_t)code, (int)e8m0 - 127 - 6);
}

/* Encode a [rows][cols] tensor (fp32, or bf16 when in_is_bf16), groups of 32 along
 * the rows: RHT32 then S2F6. codes [rows][cols], e8m0 [rows][cols/32]. */
EXPORT void orc_combine_encode(const void* in, int in_is_bf16, int64_t rows, int64_t cols,
                               uint32_t signs, uint8_t* codes, uint8_t* e8m0)
{
    float v[32];
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < cols / 32; ++g) {
            for (int i = 0; i < 32; ++i) {
                int64_t k = r * cols + g * 32 + i;
                v[i] = in_is_bf16 ? bf16_value(((const uint16_t*)in)[k]) : ((const float*)in)[k];
            }
            orc_rht32_group(v, signs);
            orc_s2f6_block(v, &codes[r * cols + g * 32], &e8m0[r * (cols / 32) + g]);
        }
}

/* Decode: token t's k arrivals are rows t*k .. t*k+k-1 of codes / e8m0; their
 * dequantized values are summed in fp32 (slot order), then rotated back.
 * out [tokens][cols] fp32. */
EXPORT void orc_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k,
                               int64_t cols, uint32_t signs, float* out)
{
    float acc[32];
    for (int64_t t = 0; t < tokens; ++t)
        for (int64_t g = 0; g < cols / 32; ++g) {
            for (int64_t j = 0; j < k; ++j) {
                int64_t r = t * k + j;
                uint8_t sc = e8m0[r * (cols / 32) + g];
                for (int i = 0; i < 32; ++i) {
                    float z = (float)orc_s2f6_decode(codes[r * cols + g * 32 + i], sc);   /* exact */
                    acc[i] = (j == 0) ? z : acc[i] + z;
                }
            }
            orc_irht32_group(acc, signs);
            for (int i = 0; i < 32; ++i) out[t * cols + g * 32 + i] = acc[i];
        }
}

/* ------------------------------------------------------------------------- */
/* MXFP4 (the Open Compute microscaling format the pages compare NVFP4 with): */
/* E2M1 codes, one E8M0 power-of-two scale per 32 consecutive values of a row. */
/* [AC] "The scaling math, worked": scale = 2^ceil(log2(amax / 6)), q =       */
/* round_to_E2M1(x / scale) (amax 22 -> scale 4, 22 -> 5.5 -> 6 -> 24);       */
/* [NV] "NVFP4 Format and Quantization Procedure" / App. B.4 on MXFP4 (a block */
/* with amax 3 + delta keeps 3 as its largest code); [NV] Section 5: MXFP4    */
/* pairs with 32-point Hadamard transforms.                                  */
/* Readings: the ceiling exponent is orc_pow2_ceil_exponent(amax, 6) (the     */
/* MXFP8 rule with the E2M1 maximum), clamped to [-127, 127]; codes are RNE   */
/* ties to even (as NVFP4); with rht the row's groups of 32 are rotated by    */
/* orc_rht32_group first (in fp32) and the rotated values are quantized.     */
/* codes [rows][cols/2] (element 2j low nibble), e8m0 [rows][cols/32].        */
/* ------------------------------------------------------------------------- */
EXPORT void orc_quantize_mxfp4(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int rht,
                               uint32_t signs, uint8_t* codes, uint8_t* e8m0)
{
    float v[32];
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < cols / 32; ++g) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_value(x[r * ld + g * 32 + i]);
            if (rht) orc_rht32_group(v, signs);
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) if (fabs((double)v[i]) > amax) amax = fabs((double)v[i]);
            int e = orc_pow2_ceil_exponent(amax, 6.0);
            e8m0[r * (cols / 32) + g] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                float t = (float)ldexp((double)v[i], -e);      /* exact power-of-two scaling */
                put_code(codes, cols / 2, r, g * 32 + i, orc_e2m1_encode_rne(t));
            }
        }
}

/* MXFP4 dequantize: code x 2^(e8m0 - 127), exact in double. */
EXPORT void orc_dequant_mxfp4(const uint8_t* codes, const uint8_t* e8m0, int64_t rows, int64_t cols,
                              double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = orc_e2m1_decode(get_code(codes, cols / 2, r, c))
                                * ldexp(1.0, (int)e8m0[r * (cols / 32) + c / 32] - 127);
}

/* ------------------------------------------------------------------------- */
/* GELU between the MLP's two linear layers                                   */
/* ------------------------------------------------------------------------- */
/* 4bit.vizuara.ai §13-14 puts GELU between the two NVFP4 linear layers of the MLP
 * block. The exact-erf GELU (Hendrycks and Gimpel, "Gaussian Error Linear Units",
 * 2016, §2): GELU(x) = x * Phi(x), Phi the standard normal cdf, and its derivative
 * GELU'(x) = Phi(x) + x * phi(x), phi the standard normal density. Phi is written
 * through the complementary error function, Phi(x) = erfc(-x / sqrt 2) / 2, which
 * loses nothing in the lower tail (1 + erf(x / sqrt 2) cancels for x < -4). Double
 * precision throughout; libm's erfc and exp are the library steps. */
EXPORT double orc_normal_cdf(double x)
{
    return 0.5 * erfc(-x / sqrt(2.0));
}

EXPORT double orc_normal_pdf(double x)
{
    return exp(-0.5 * x * x) / sqrt(2.0 * 3.14159265358979323846);
}

EXPORT double orc_gelu(double x)
{
    return x * orc_normal_cdf(x);
}

EXPORT double orc_gelu_grad(double x)
{
    return orc_normal_cdf(x) + x * orc_normal_pdf(x);
}

/* GELU (grad == 0) or GELU' (grad != 0) of n bf16 values, in double. */
EXPORT void orc_gelu_bf16(const uint16_t* h, int64_t n, int grad, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        const double x = (double)bf16_value(h[i]);
        out[i] = grad ? orc_gelu_grad(x) : orc_gelu(x);
    }
}
