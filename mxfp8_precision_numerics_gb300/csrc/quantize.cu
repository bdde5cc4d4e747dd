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

// Block scale code and the local encode scale (steps 2-3).
__device__ __forceinline__ uint32_t block_scale(float amax_b, float s_enc) {
    float v = __fmul_rn(__fdiv_rn(amax_b, 6.0f), s_enc);
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

}  // namespace fp4q
