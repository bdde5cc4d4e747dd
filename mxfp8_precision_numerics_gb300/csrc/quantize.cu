// quantize.cu — per-tensor amax and NVFP4 1D (1x16) / 2D (16x16) quantization kernels.
//
// "Pretraining Large Language Models with NVFP4", "NVFP4 Format and Quantization
// Procedure", steps 1-4 (two-level scaling), and "Two-Dimensional Weight Scaling and the
// Chain Rule Problem" (one scale per 16x16 weight tile); 4bit.vizuara.ai §5-6 and §13.
//
// Both kernels are HBM-bound streams. The amax pass reads the bf16 tensor once with
// 16-byte loads and reduces |x| as integers (the magnitude order of non-NaN bf16 equals
// the order of their low 15 bits), sweeping the address range front to back. The quantize
// pass reads it again back to front (so the part still in L2 is read first), 32 bytes (one
// 16-value block) per thread, and writes 8 bytes of codes and 1 scale byte per block.
#include "fp4q_common.cuh"
#include "fp4q_internal.h"

namespace fp4q {

// ---------------------------------------------------------------------------------------
// amax over a [rows][ld] bf16 tensor (cols used per row), `batch` tensors along blockIdx.y.
// The tensor is walked in 4 KB row segments (256 16-byte vectors), segment u by warp
// u mod W in round u div W, so the segments in flight at any time are adjacent in memory and
// the pass sweeps the address range once; the quantize pass then walks it backwards and
// finds the most recently read part still in L2.
// out[b] must be zero before the launch (atomicMax on the fp32 bit pattern).
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x,
                                                        int64_t rows, int64_t cols, int64_t ld,
                                                        int64_t batch_stride,
                                                        float* __restrict__ out) {
    const uint16_t* base = x + (int64_t)blockIdx.y * batch_stride;
    const int64_t vecs = cols / 8;
    const int64_t segs = (vecs + 255) / 256;
    const int64_t units = rows * segs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * 8;
    uint32_t m2 = 0;   // two packed |bf16| maxima
    for (int64_t u = (int64_t)blockIdx.x * 8 + warp; u < units; u += warps_total) {
        const int64_t r = u / segs, sg = u - r * segs;
        const uint4* row = reinterpret_cast<const uint4*>(base + r * ld);
        const int64_t v0 = sg * 256, v1 = v0 + 256 < vecs ? v0 + 256 : vecs;
        if (v1 - v0 == 256) {
            uint4 q[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) q[k] = __ldg(row + v0 + lane + 32 * k);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(q[k].x & 0x7FFF7FFFu, q[k].y & 0x7FFF7FFFu),
                                           __vmaxu2(q[k].z & 0x7FFF7FFFu, q[k].w & 0x7FFF7FFFu)));
        } else {
            for (int64_t v = v0 + lane; v < v1; v += 32) {
                uint4 a = __ldg(row + v);
                m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                           __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
            }
        }
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __shared__ uint32_t red[8];
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) t = max(t, red[i]);
        // bf16 magnitude bits << 16 is the fp32 bit pattern of the same value
        atomicMax(reinterpret_cast<unsigned int*>(out + blockIdx.y), t << 16);
    }
}

// Per-tensor scales from the amax ("NVFP4 Format and Quantization Procedure", step 1):
// s_enc = 2688 / amax, s_dec = 1 / s_enc; amax == 0 or a non-finite s_enc gives 1 and 1.
__device__ __forceinline__ void global_scales(float amax, float& s_enc, float& s_dec) {
    s_enc = __fdiv_rn(2688.0f, amax);
    if (!(amax > 0.0f) || !isfinite(s_enc)) s_enc = 1.0f;
    s_dec = __fdiv_rn(1.0f, s_enc);
}

// amax_b / 6 correctly rounded, for amax_b a non-negative bf16 value: q0 = amax_b * RN(1/6), then
// one fused multiply-add correction, q0 + RN(amax_b - 6 q0) * RN(1/6) (division by a constant
// with a correction step, Brisebarre, Muller and Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance", IEEE TC 2004). Equal to the
// IEEE quotient for every one of the 32640 non-negative finite bf16 values (checked exhaustively
// in exact arithmetic by the CPU tests).
__device__ __forceinline__ float div6_bf16(float a) {
    const float c = 0.16666667163372039795f;   // RN(1/6) = 0x3E2AAAAB
    const float q0 = __fmul_rn(a, c);
    const float r = __fmaf_rn(-q0, 6.0f, a);
    return __fmaf_rn(r, c, q0);
}

// Block scale code and the local encode scale (steps 2-3); amax_b is a bf16 value.
__device__ __forceinline__ uint32_t block_scale(float amax_b, float s_enc) {
    float v = __fmul_rn(div6_bf16(amax_b), s_enc);
    uint32_t sb = e4m3_rne_sat(v) & 0x7Fu;
    return sb == 0 ? 1u : sb;
}

__device__ __forceinline__ float block_encode_scale(uint32_t sb, float s_dec) {
    return __fdiv_rn(1.0f, __fmul_rn(e4m3_to_f32(sb), s_dec));
}

// 16 bf16 (as 8 packed words) -> 16 E2M1 codes packed into 64 bits (element 2j low nibble).
template <bool kHwCvt>
__device__ __forceinline__ uint2 encode16(const uint32_t (&w)[8], float s_enc_b) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a = __fmul_rn(__uint_as_float(w[j] << 16), s_enc_b);
        float b = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), s_enc_b);
        uint32_t byte = kHwCvt ? e2m1x2_cvt_rn(a, b) : (e2m1_rne_alu(a) | (e2m1_rne_alu(b) << 4));
        if (j < 4) lo |= byte << (8 * j); else hi |= byte << (8 * (j - 4));
    }
    return make_uint2(lo, hi);
}

__device__ __forceinline__ float absmax16(const uint32_t (&w)[8]) {
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m2 = __vmaxu2(m2, w[j] & 0x7FFF7FFFu);
    return __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
}

// ---------------------------------------------------------------------------------------
// 1D quantize: one thread per 16-value block. amax comes from amax_src (device float).
// ---------------------------------------------------------------------------------------
template <bool kHwCvt>
__global__ void __launch_bounds__(256) quantize_1d_kernel(const uint16_t* __restrict__ x,
                                                          int64_t rows, int64_t cols, int64_t ld,
                                                          const float* __restrict__ amax_src,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales,
                                                          float* __restrict__ s_dec_out) {
    const int64_t nb = cols >> 4;
    const int64_t total = rows * nb;
    float s_enc, s_dec;
    global_scales(*amax_src, s_enc, s_dec);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        // last rows first: they are the ones the amax pass read most recently, still in L2
        const int64_t b = total - 1 - i;
        const int64_t r = b / nb, j = b - r * nb;
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + j * 16);
        uint4 p = __ldcs(src), q = __ldcs(src + 1);
        uint32_t w[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
        uint32_t sb = block_scale(absmax16(w), s_enc);
        uint2 c = encode16<kHwCvt>(w, block_encode_scale(sb, s_dec));
        reinterpret_cast<uint2*>(codes)[b] = c;   // codes row = cols/2 bytes = nb * 8
        scales[b] = (uint8_t)sb;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_dec_out = s_dec;
}

// ---------------------------------------------------------------------------------------
// 2D quantize: a CTA covers 16 rows x (256 kQ2Tiles) columns (16 kQ2Tiles tiles of 16x16).
// Thread (r, t) loads row r of tiles t, t+16, ... (kQ2Tiles 32-byte loads in flight; 16
// consecutive threads cover 512 contiguous bytes of one row per load), the tile amax is
// reduced through shared memory, then each thread encodes its values with their tiles'
// scales. blockIdx.z = batch index (one tensor per expert).
// ---------------------------------------------------------------------------------------
constexpr int kQ2Tiles = 2;

template <bool kHwCvt>
__global__ void __launch_bounds__(256) quantize_2d_kernel(const uint16_t* __restrict__ w,
                                                          int64_t rows, int64_t cols, int64_t ld,
                                                          int64_t batch_stride,
                                                          const float* __restrict__ amax_src,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ tile_scales,
                                                          float* __restrict__ s_dec_out) {
    const int bz = blockIdx.z;
    const int r = threadIdx.x >> 4, t = threadIdx.x & 15;
    const int64_t tcols = cols >> 4;
    // last row strips first (the amax pass read them most recently; they are still in L2)
    const int64_t by = (int64_t)gridDim.y - 1 - blockIdx.y;
    const int64_t row = by * 16 + r;
    float s_enc, s_dec;
    global_scales(amax_src[bz], s_enc, s_dec);
    uint32_t v[kQ2Tiles][8];
    bool valid[kQ2Tiles];
#pragma unroll
    for (int h = 0; h < kQ2Tiles; ++h) {
        const int64_t tile_c = (int64_t)blockIdx.x * (16 * kQ2Tiles) + 16 * h + t;
        valid[h] = tile_c < tcols;
#pragma unroll
        for (int k = 0; k < 8; ++k) v[h][k] = 0;
        if (valid[h]) {
            const uint4* src = reinterpret_cast<const uint4*>(w + bz * batch_stride + row * ld + tile_c * 16);
            uint4 p = __ldcs(src), q = __ldcs(src + 1);
            v[h][0] = p.x; v[h][1] = p.y; v[h][2] = p.z; v[h][3] = p.w;
            v[h][4] = q.x; v[h][5] = q.y; v[h][6] = q.z; v[h][7] = q.w;
        }
    }
    __shared__ float part[kQ2Tiles][16][17];
#pragma unroll
    for (int h = 0; h < kQ2Tiles; ++h) part[h][r][t] = absmax16(v[h]);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kQ2Tiles; ++h) {
        float amax_b = part[h][0][t];
#pragma unroll
        for (int i = 1; i < 16; ++i) amax_b = fmaxf(amax_b, part[h][i][t]);
        if (valid[h]) {
            const int64_t tile_c = (int64_t)blockIdx.x * (16 * kQ2Tiles) + 16 * h + t;
            uint32_t sb = block_scale(amax_b, s_enc);
            uint2 c = encode16<kHwCvt>(v[h], block_encode_scale(sb, s_dec));
            uint8_t* crow = codes + bz * (rows * (cols >> 1)) + row * (cols >> 1);
            reinterpret_cast<uint2*>(crow)[tile_c] = c;
            if (r == 0) tile_scales[bz * ((rows >> 4) * tcols) + by * tcols + tile_c] = (uint8_t)sb;
        }
    }
    if (blockIdx.x == 0 && by == 0 && threadIdx.x == 0) s_dec_out[bz] = s_dec;
}

// ---------------------------------------------------------------------------------------
// 1D quantize with one outer scale per row and, optionally, the Four Over Six block scale
// (4bit.vizuara.ai §10; "End-to-End 4-Bit Training" (Thinking Machines), 方案细节).
// One pass over HBM and no amax kernel: a row's blocks are loaded into registers (kHold
// blocks of 16 per thread, 1, 2 or 4; a longer row reads the rest again, from L2), the row
// amax is reduced across the row's threads, and the blocks are encoded from registers.
// A row is handled by W warps (W = 1, 2, 4 or 8), 8 / W rows per 256-thread CTA; thread t
// of a row owns blocks t, t + 32W, t + 64W, ... so each load instruction of a warp covers
// 512 contiguous bytes.
// ---------------------------------------------------------------------------------------
constexpr int kRowHoldMax = 4;

// The low bytes of a, b, c, d as one word (a lowest): three byte permutes.
__device__ __forceinline__ uint32_t pack_bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// Two fp32 values (a packed pair) -> their E2M1 codes (one byte, low nibble = low half, round
// to nearest even, saturating) and the grid values of those codes as a packed fp32 pair.
__device__ __forceinline__ uint32_t e2m1x2_roundtrip(uint64_t y2, uint64_t& q2) {
    uint32_t byte;
    asm("{.reg .b8 t; .reg .b32 h; .reg .f32 y0, y1, a, b; .reg .f16 l, u;\n\t"
        "mov.b64 {y0, y1}, %2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, y1, y0;\n\t"
        "cvt.rn.f16x2.e2m1x2 h, t;\n\t"
        "mov.b32 {l, u}, h;\n\t"
        "cvt.f32.f16 a, l;\n\t"
        "cvt.f32.f16 b, u;\n\t"
        "mov.b64 %1, {a, b};\n\t"
        "cvt.u32.u8 %0, t;}"
        : "=r"(byte), "=l"(q2) : "l"(y2));
    return byte;
}

// The 16 values of a block (8 packed bf16 words) encoded with both Four Over Six candidates
// (local encode scales se6 and se4): codes c6 / c4 and, for each, the sum of squared
// distances between the scaled values y and their grid points q. y - q is exact; the squares
// go into two fused multiply-add chains, one over the even positions and one over the odd
// (the two halves of packed fp32 pairs), which are added at the end.
__device__ __forceinline__ void encode16_46(const uint32_t (&w)[8], float se6, float se4, uint2& c6, uint2& c4,
                                            float& sq6, float& sq4) {
    uint64_t s6, s4, a6, a4;
    asm("mov.b64 %0, {%1, %1};" : "=l"(s6) : "f"(se6));
    asm("mov.b64 %0, {%1, %1};" : "=l"(s4) : "f"(se4));
    asm("mov.b64 %0, {%1, %1};" : "=l"(a6) : "f"(0.0f));
    a4 = a6;
    uint32_t b6[8], b4[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint64_t x2, y6, y4, q6, q4, d6, d4;
        asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "r"(w[j] << 16), "r"(w[j] & 0xFFFF0000u));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y6) : "l"(x2), "l"(s6));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y4) : "l"(x2), "l"(s4));
        b6[j] = e2m1x2_roundtrip(y6, q6);
        b4[j] = e2m1x2_roundtrip(y4, q4);
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d6) : "l"(y6), "l"(q6));
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d4) : "l"(y4), "l"(q4));
        asm("fma.rn.f32x2 %0, %1, %1, %0;" : "+l"(a6) : "l"(d6));
        asm("fma.rn.f32x2 %0, %1, %1, %0;" : "+l"(a4) : "l"(d4));
    }
    float e0, e1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(e0), "=f"(e1) : "l"(a6));
    sq6 = __fadd_rn(e0, e1);
    asm("mov.b64 {%0, %1}, %2;" : "=f"(e0), "=f"(e1) : "l"(a4));
    sq4 = __fadd_rn(e0, e1);
    c6 = make_uint2(pack_bytes4(b6[0], b6[1], b6[2], b6[3]), pack_bytes4(b6[4], b6[5], b6[6], b6[7]));
    c4 = make_uint2(pack_bytes4(b4[0], b4[1], b4[2], b4[3]), pack_bytes4(b4[4], b4[5], b4[6], b4[7]));
}

// Both candidate block scales from one hardware conversion (round to nearest even, saturating
// at 448: the rule of e4m3_rne_sat): byte 0 for target 6, (amax_b / 6) * s_enc, and byte 1 for
// target 4, (amax_b / 4) * s_enc; a scale that rounds to zero is raised to the smallest code.
__device__ __forceinline__ uint32_t scale_codes_46(float amax_b, float s_enc) {
    const float v6 = __fmul_rn(div6_bf16(amax_b), s_enc);
    const float v4 = __fmul_rn(__fmul_rn(amax_b, 0.25f), s_enc);     // amax_b / 4 is exact
    uint32_t c;
    asm("{.reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t;}" : "=r"(c) : "f"(v4), "f"(v6));
    return __vmaxu4(c, 0x0101u);
}

// The low two bytes of c as E4M3 values in fp32 (exact through f16).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t c, float& lo, float& hi) {
    asm("{.reg .b16 t; .reg .b32 h; .reg .f16 l, u;\n\t"
        "cvt.u16.u32 t, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, t;\n\t"
        "mov.b32 {l, u}, h;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, u;}"
        : "=f"(lo), "=f"(hi) : "r"(c));
}

template <bool kFourSix>
__device__ __forceinline__ void encode_row_block(const uint32_t (&w)[8], float s_enc, float s_dec,
                                                 uint8_t* crow, uint8_t* srow, int64_t b) {
    const float amax_b = absmax16(w);
    uint32_t sb;
    uint2 c;
    if (!kFourSix) {
        sb = block_scale(amax_b, s_enc);
        c = encode16<true>(w, block_encode_scale(sb, s_dec));
    } else {
        const uint32_t sc = scale_codes_46(amax_b, s_enc);
        float S6, S4;
        e4m3x2_to_f32(sc, S6, S4);
        uint2 c4;
        float sq6, sq4;
        encode16_46(w, __frcp_rn(__fmul_rn(S6, s_dec)), __frcp_rn(__fmul_rn(S4, s_dec)), c, c4, sq6, sq4);
        const float e6 = __fmul_rn(sq6, __fmul_rn(S6, S6)), e4 = __fmul_rn(sq4, __fmul_rn(S4, S4));
        sb = sc & 0xFFu;
        if (e4 < e6) {   // a tie keeps the ordinary scale
            sb = (sc >> 8) & 0xFFu;
            c = c4;
        }
    }
    reinterpret_cast<uint2*>(crow)[b] = c;
    srow[b] = (uint8_t)sb;
}

__device__ __forceinline__ void load_block(const uint16_t* xr, int64_t b, bool stream, uint32_t (&w)[8]) {
    const uint4* src = reinterpret_cast<const uint4*>(xr + b * 16);
    const uint4 p = stream ? __ldcs(src) : __ldg(src), q = stream ? __ldcs(src + 1) : __ldg(src + 1);
    w[0] = p.x; w[1] = p.y; w[2] = p.z; w[3] = p.w;
    w[4] = q.x; w[5] = q.y; w[6] = q.z; w[7] = q.w;
}

template <bool kFourSix, int kHold>
__global__ void __launch_bounds__(256) quantize_1d_rows_kernel(const uint16_t* __restrict__ x,
                                                               int64_t rows, int64_t cols, int64_t ld, int W,
                                                               uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ scales,
                                                               float* __restrict__ s_dec_rows) {
    const int T = 32 * W;
    const int lr = threadIdx.x / T, t = threadIdx.x - lr * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (8 / W) + lr;
    const bool row_ok = row < rows;
    const int64_t nb = cols >> 4;
    const uint16_t* xr = x + (row_ok ? row : 0) * ld;

    uint32_t w[kHold][8];
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
        const int64_t b = t + (int64_t)j * T;
        if (row_ok && b < nb) {
            load_block(xr, b, true, w[j]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) w[j][k] = 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) m2 = __vmaxu2(m2, w[j][k] & 0x7FFF7FFFu);
    }
    for (int64_t b = t + (int64_t)kHold * T; row_ok && b < nb; b += T) {   // rows longer than held
        uint32_t v[8];
        load_block(xr, b, false, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) m2 = __vmaxu2(m2, v[k] & 0x7FFF7FFFu);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __shared__ uint32_t red[8];
    if (lane == 0) red[warp] = m;
    __syncthreads();
    for (int i = 0; i < W; ++i) m = max(m, red[lr * W + i]);
    if (!row_ok) return;
    float s_enc, s_dec;
    global_scales(__uint_as_float(m << 16), s_enc, s_dec);   // |bf16| bits << 16 = its fp32 pattern

    uint8_t* crow = codes + row * (cols >> 1);
    uint8_t* srow = scales + row * nb;
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
        const int64_t b = t + (int64_t)j * T;
        if (b < nb) encode_row_block<kFourSix>(w[j], s_enc, s_dec, crow, srow, b);
    }
    for (int64_t b = t + (int64_t)kHold * T; b < nb; b += T) {
        uint32_t v[8];
        load_block(xr, b, true, v);
        encode_row_block<kFourSix>(v, s_enc, s_dec, crow, srow, b);
    }
    if (t == 0) s_dec_rows[row] = s_dec;
}

// ---------------------------------------------------------------------------------------
// host launchers (validated by the C-ABI layer)
// ---------------------------------------------------------------------------------------
static int grid_for(int64_t work_items, int threads) {
    int64_t g = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 16;   // 16 resident 256-thread CTAs per SM at most
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                        int64_t batch_stride, float* out, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * batch, st);
    if (e != cudaSuccess) return e;
    const int64_t units = rows * ((cols / 8 + 255) / 256);
    int64_t g = (units + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    amax_bf16_kernel<<<dim3((unsigned)g, (unsigned)batch), 256, 0, st>>>(x, rows, cols, ld,
                                                                         batch_stride, out);
    return cudaGetLastError();
}

cudaError_t launch_quantize_1d(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                               const float* amax, uint8_t* codes, uint8_t* scales, float* s_dec,
                               cudaStream_t st) {
    int64_t items = rows * (cols / 16);
    int g = grid_for(items, 256);
    if (use_hw_e2m1())
        quantize_1d_kernel<true><<<g, 256, 0, st>>>(x, rows, cols, ld, amax, codes, scales, s_dec);
    else
        quantize_1d_kernel<false><<<g, 256, 0, st>>>(x, rows, cols, ld, amax, codes, scales, s_dec);
    return cudaGetLastError();
}

cudaError_t launch_quantize_2d(const uint16_t* w, int64_t rows, int64_t cols, int64_t ld,
                               int64_t batch, int64_t batch_stride, const float* amax,
                               uint8_t* codes, uint8_t* tile_scales, float* s_dec,
                               cudaStream_t st) {
    dim3 grid((unsigned)((cols / 16 + 16 * kQ2Tiles - 1) / (16 * kQ2Tiles)), (unsigned)(rows / 16), (unsigned)batch);
    if (use_hw_e2m1())
        quantize_2d_kernel<true><<<grid, 256, 0, st>>>(w, rows, cols, ld, batch_stride, amax, codes,
                                                       tile_scales, s_dec);
    else
        quantize_2d_kernel<false><<<grid, 256, 0, st>>>(w, rows, cols, ld, batch_stride, amax, codes,
                                                        tile_scales, s_dec);
    return cudaGetLastError();
}

// Warps per row and blocks held per thread: up to 4 blocks per thread (a load of 128 bytes
// per thread in flight before the row's amax is known) and as few warps as cover the row, up
// to 8; a row longer than 8 warps x 4 blocks reads the rest twice.
void rows_shape(int64_t cols, int& W, int& hold) {
    const int64_t nb = cols / 16;
    W = 1;
    while (W < 8 && (int64_t)32 * W * kRowHoldMax < nb) W *= 2;
    hold = 1;
    while (hold < kRowHoldMax && (int64_t)32 * W * hold < nb) hold *= 2;
}

template <bool kFourSix>
static void launch_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int W, int hold,
                        uint8_t* codes, uint8_t* scales, float* s_dec_rows, unsigned g, cudaStream_t st) {
    if (hold == 1)
        quantize_1d_rows_kernel<kFourSix, 1><<<g, 256, 0, st>>>(x, rows, cols, ld, W, codes, scales, s_dec_rows);
    else if (hold == 2)
        quantize_1d_rows_kernel<kFourSix, 2><<<g, 256, 0, st>>>(x, rows, cols, ld, W, codes, scales, s_dec_rows);
    else
        quantize_1d_rows_kernel<kFourSix, 4><<<g, 256, 0, st>>>(x, rows, cols, ld, W, codes, scales, s_dec_rows);
}

cudaError_t launch_quantize_1d_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int four_six,
                                    uint8_t* codes, uint8_t* scales, float* s_dec_rows, cudaStream_t st) {
    int W, hold;
    rows_shape(cols, W, hold);
    const int64_t g = (rows + (8 / W) - 1) / (8 / W);
    if (g > 2147483647) return cudaErrorInvalidValue;
    if (four_six)
        launch_rows<true>(x, rows, cols, ld, W, hold, codes, scales, s_dec_rows, (unsigned)g, st);
    else
        launch_rows<false>(x, rows, cols, ld, W, hold, codes, scales, s_dec_rows, (unsigned)g, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// MXFP4 quantize ("FP4 Training on Blackwell", "The scaling math, worked"; the format the
// NVFP4 paper compares against): E2M1 codes with one E8M0 scale per 32 values of a row,
// scale 2^e with e the smallest integer such that amax <= 6 * 2^e (clamped to [-127, 127]).
// One thread per group of 32 (four 16-byte loads), optionally rotated by RHT32 first (the
// 32-point transform the paper pairs with MXFP4); codes by the hardware E2M1 conversion of the
// exactly scaled values; 16 code bytes and one scale byte per thread. (A variant that staged
// 32-group chunks per warp through shared memory by cp.async measured 6-8% slower: this
// kernel's loads already keep HBM busy and its arithmetic, not memory, is the limit with RHT.)
// ---------------------------------------------------------------------------------------
// 6 = 1.5 * 2^2: amax = m 2^E (m in [1, 2)) -> e = E - 2 + (m > 1.5); subnormal amax -> -127;
// an infinite amax satisfies no e and takes the clamp, 127.
__device__ __forceinline__ int mxfp4_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (u < 0x00800000u) return -127;
    if (u >= 0x7F800000u) return 127;
    const int e = (int)(u >> 23) - 127 - 2 + ((u & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// encode one group of 32 (already rotated if kRht): E2M1 codes (4 words) and the E8M0 byte
template <bool kRht>
__device__ __forceinline__ uint32_t mxfp4_group(float (&v)[32], uint32_t signs, uint32_t (&out)[4]) {
    if (kRht) rht32_forward(v, signs);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mxfp4_exponent(amax);
    const float inv = exp2i(-e);          // v * 2^-e is exact (|result| <= 6)
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b[j] = e2m1x2_cvt_rn(__fmul_rn(v[8 * wd + 2 * j], inv), __fmul_rn(v[8 * wd + 2 * j + 1], inv));
        out[wd] = pack_bytes4(b[0], b[1], b[2], b[3]);
    }
    return (uint32_t)(e + 127);
}

template <bool kRht>
__global__ void __launch_bounds__(256) quantize_mxfp4_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int64_t cols, int64_t ld, uint32_t signs,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ e8m0) {
    const int64_t gpr = cols >> 5;
    const int64_t groups = rows * gpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const int64_t r = g / gpr, c = g - r * gpr;
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + c * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 p = __ldcs(src + q);
            const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[8 * q + 2 * k] = __uint_as_float(w[k] << 16);
                v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
        }
        uint32_t out[4];
        const uint32_t sc = mxfp4_group<kRht>(v, signs, out);
        __stcs(reinterpret_cast<uint4*>(codes + r * (cols >> 1) + c * 16), make_uint4(out[0], out[1], out[2], out[3]));
        e8m0[g] = (uint8_t)sc;
    }
}

cudaError_t launch_quantize_mxfp4(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int rht, uint32_t signs,
                                  uint8_t* codes, uint8_t* e8m0, cudaStream_t st) {
    const int g = grid_for(rows * (cols / 32), 256);
    if (rht)
        quantize_mxfp4_kernel<true><<<g, 256, 0, st>>>(x, rows, cols, ld, signs, codes, e8m0);
    else
        quantize_mxfp4_kernel<false><<<g, 256, 0, st>>>(x, rows, cols, ld, signs, codes, e8m0);
    return cudaGetLastError();
}

}  // namespace fp4q
