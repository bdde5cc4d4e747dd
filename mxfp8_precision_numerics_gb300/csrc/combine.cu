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
// Kernels (HBM streams; one lane per group of 32 values):
//   combine_encode_staged  fp32 [rows][cols] -> S2F6 bytes [rows][cols] + E8M0 [rows][cols/32]
//   combine_encode_kernel  the same from bf16, one thread per group, grid-stride (with half the
//                          input bytes per group the arithmetic, not the bytes in flight, is
//                          the limit, and staging measured slower)
//   combine_decode_staged  k arrivals per token (rows t*k .. t*k+k-1) -> their sum rotated back,
//                          fp32 or bf16 [tokens][cols]; used when cols % 1024 == 0, the E8M0
//                          pointer is 4-byte aligned and the ring fits in 227 KB (k <= 7 for
//                          fp32 output, k <= 8 for bf16)
//   combine_decode_kernel  the same for every other shape (one thread per group, grid-stride)
// The staged kernels give each warp a chunk of 32 consecutive groups at a time (warp w takes
// chunks w, w + W, ...). A chunk's input reaches the warp's shared-memory ring by cp.async
// kStages - 1 chunks ahead, as coalesced 16-byte pieces placed with an XOR swizzle so that
// each lane, reading its own group's pieces, hits distinct banks; outputs wider than 16
// bytes per lane leave through shared memory the same way, as coalesced 16-byte stores.
// The bytes in flight per SM are then set by the ring, not by the registers.
// The conversion instructions for block-scaled S2F6 that the pages list are not accepted by
// this toolkit's assembler for sm_103a; the codes are formed with fp32 adds and byte permutes
// instead (s2f6_encode32 / s2f6_decode4).
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

constexpr int kChunk = 32;            // groups per warp chunk (one per lane)

// Byte offset of 16-byte piece q of group gr in a chunk whose groups are `pieces` pieces
// long (2, 4 or 8): any 8 consecutive lanes reading piece q of their own groups, and any 8
// consecutive pieces of the chunk in order, fall in 8 distinct 16-byte bank slots.
__device__ __forceinline__ uint32_t chunk_off(int gr, int q, int pieces) {
    const int sh = pieces == 8 ? 0 : (pieces == 4 ? 1 : 2);
    return (uint32_t)(gr * pieces * 16 + ((q ^ ((gr >> sh) & (pieces - 1))) * 16));
}

template <bool kBf16, int kStages>
__global__ void __launch_bounds__(256) combine_encode_staged(const void* __restrict__ in, int64_t groups,
                                                             uint32_t signs, uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ e8m0) {
    constexpr int kP = kBf16 ? 4 : 8;                     // input pieces per group
    constexpr int kIn = kChunk * kP * 16;                 // input bytes per chunk
    constexpr int kWarpBytes = kStages * kIn + kChunk * 32;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * kWarpBytes;
    uint8_t* obuf = ring + kStages * kIn;
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    const uint8_t* src = static_cast<const uint8_t*>(in);
    const int64_t nchunks = (groups + kChunk - 1) / kChunk;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
    auto issue = [&](int64_t n, int slot) {
#pragma unroll
        for (int i = 0; i < kP; ++i) {
            const int p = lane + 32 * i, gr = p / kP, q = p % kP;
            const int64_t g = n * kChunk + gr;
            const bool ok = g < groups;
            cp_async16(ring_s + slot * kIn + chunk_off(gr, q, kP), src + (ok ? g * (kP * 16) + q * 16 : 0), ok);
        }
    };
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) {
        if (w0 + t * nw < nchunks) issue(w0 + t * nw, t);
        cp_async_commit();
    }
    int slot = 0;
    for (int64_t n = w0; n < nchunks; n += nw) {
        const int64_t nn = n + (int64_t)(kStages - 1) * nw;
        if (nn < nchunks) issue(nn, (slot + kStages - 1) % kStages);
        cp_async_commit();
        cp_async_wait<kStages - 1>();                      // chunk n has landed (own pieces)
        __syncwarp();                                      // ... and every lane's
        const uint8_t* st = ring + slot * kIn;
        float v[32];
        if (kBf16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w4 = *reinterpret_cast<const uint4*>(st + chunk_off(lane, q, 4));
                const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * q + 2 * k] = __uint_as_float(w[k] << 16);
                    v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 f = *reinterpret_cast<const float4*>(st + chunk_off(lane, q, 8));
                v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
            }
        }
        rht32_forward(v, signs);
        uint32_t out[8];
        const uint32_t sc = s2f6_encode32(v, out);
        *reinterpret_cast<uint4*>(obuf + chunk_off(lane, 0, 2)) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(obuf + chunk_off(lane, 1, 2)) = make_uint4(out[4], out[5], out[6], out[7]);
        if (n * kChunk + lane < groups) e8m0[n * kChunk + lane] = (uint8_t)sc;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int p = lane + 32 * i, gr = p >> 1, q = p & 1;
            if (n * kChunk + gr < groups)
                __stcs(reinterpret_cast<uint4*>(codes + (n * kChunk + gr) * 32 + q * 16),
                       *reinterpret_cast<const uint4*>(obuf + chunk_off(gr, q, 2)));
        }
        __syncwarp();                                      // ring slot and obuf free again
        slot = slot + 1 == kStages ? 0 : slot + 1;
    }
    cp_async_wait<0>();
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

// Decode, staged: chunk n is 32 groups of one token t (cols % 1024 == 0), starting at
// column group c0; its slot holds the k arrivals' 1 KB of codes each (swizzled as 2-piece
// groups) and then their 32 scale bytes each.
template <bool kOutBf16, int kStages>
__global__ void __launch_bounds__(256, 3) combine_decode_staged(const uint8_t* __restrict__ codes,
                                                             const uint8_t* __restrict__ e8m0,
                                                             int64_t tokens, int k, int64_t gpr,
                                                             uint32_t signs, void* __restrict__ out) {
    constexpr int kOutP = kOutBf16 ? 4 : 8;                // output pieces per group
    extern __shared__ __align__(16) uint8_t smem[];
    const int slot_bytes = k * (1024 + 32);
    const int warp_bytes = kStages * slot_bytes + kChunk * kOutP * 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * warp_bytes;
    uint8_t* obuf = ring + kStages * slot_bytes;
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    const int64_t nchunks = tokens * gpr / kChunk;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
    auto issue = [&](int64_t n, int slot) {
        const int64_t g0 = n * kChunk, t = g0 / gpr, c0 = g0 - t * gpr, row0 = t * k;
        const uint32_t base = ring_s + slot * slot_bytes;
        for (int i = 0; i < 2 * k; ++i) {                 // k x 64 code pieces
            const int p = lane + 32 * i, j = p >> 6, gr = (p & 63) >> 1, q = p & 1;
            cp_async16(base + j * 1024 + chunk_off(gr, q, 2), codes + ((row0 + j) * gpr + c0 + gr) * 32 + q * 16, true);
        }
        for (int p = lane; p < 8 * k; p += 32) {          // k x 8 scale words
            const int j = p >> 3, wd = p & 7;
            cp_async4(base + k * 1024 + j * 32 + wd * 4, e8m0 + (row0 + j) * gpr + c0 + wd * 4);
        }
    };
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) {
        if (w0 + t * nw < nchunks) issue(w0 + t * nw, t);
        cp_async_commit();
    }
    int slot = 0;
    for (int64_t n = w0; n < nchunks; n += nw) {
        const int64_t nn = n + (int64_t)(kStages - 1) * nw;
        if (nn < nchunks) issue(nn, (slot + kStages - 1) % kStages);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint8_t* st = ring + slot * slot_bytes;
        float acc[32];
        for (int j = 0; j < k; ++j) {                      // arrivals in slot order
            const uint4 a = *reinterpret_cast<const uint4*>(st + j * 1024 + chunk_off(lane, 0, 2));
            const uint4 b = *reinterpret_cast<const uint4*>(st + j * 1024 + chunk_off(lane, 1, 2));
            const uint32_t sc = st[k * 1024 + j * 32 + lane];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            if (j == 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q) s2f6_decode4(w[q], sc, acc + 4 * q);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float z[4];
                    s2f6_decode4(w[q], sc, z);
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc[4 * q + m] = __fadd_rn(acc[4 * q + m], z[m]);
                }
            }
        }
        rht32_inverse(acc, signs);
        if (kOutBf16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * q + 2 * m], acc[8 * q + 2 * m + 1]);
                    w[m] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(obuf + chunk_off(lane, q, 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(obuf + chunk_off(lane, q, 8)) =
                    make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
        __syncwarp();
        uint8_t* dst = static_cast<uint8_t*>(out) + n * kChunk * (kOutP * 16);
#pragma unroll
        for (int i = 0; i < kOutP; ++i) {
            const int p = lane + 32 * i, gr = p / kOutP, q = p % kOutP;
            __stcs(reinterpret_cast<uint4*>(dst + gr * (kOutP * 16) + q * 16),
                   *reinterpret_cast<const uint4*>(obuf + chunk_off(gr, q, kOutP)));
        }
        __syncwarp();
        slot = slot + 1 == kStages ? 0 : slot + 1;
    }
    cp_async_wait<0>();
}

static unsigned combine_grid(int64_t groups) {
    int64_t g = (groups + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

// Persistent grid for a staged kernel: resident CTAs per SM x SMs, at most one warp per chunk.
// The shared-memory opt-in and the occupancy are taken once per (kernel, bytes, device).
template <typename K>
static cudaError_t staged_grid(K kern, int smem, int64_t nchunks, unsigned* grid) {
    struct Entry { const void* fn; int smem, dev, per; };
    static Entry seen[16];
    static int n_seen = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int per = 0;
    for (int i = 0; i < n_seen; ++i)
        if (seen[i].fn == (const void*)kern && seen[i].smem == smem && seen[i].dev == dev) per = seen[i].per;
    if (per == 0) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, 256, smem)) != cudaSuccess) return e;
        if (per < 1) per = 1;
        if (n_seen < 16) seen[n_seen++] = Entry{(const void*)kern, smem, dev, per};
    }
    int64_t g = (int64_t)num_sms() * per;
    const int64_t need = (nchunks + 7) / 8;
    if (g > need) g = need;
    *grid = (unsigned)(g < 1 ? 1 : g);
    return cudaSuccess;
}

cudaError_t launch_combine_encode(const void* in, int in_bf16, int64_t rows, int64_t cols, uint32_t signs,
                                  uint8_t* codes, uint8_t* e8m0, cudaStream_t st) {
    const int64_t groups = rows * (cols / 32);
    const int64_t nchunks = (groups + kChunk - 1) / kChunk;
    unsigned g = 0;
    cudaError_t e;
    if (in_bf16) {
        combine_encode_kernel<true><<<combine_grid(groups), 256, 0, st>>>(in, groups, signs, codes, e8m0);
    } else {
        constexpr int kS = 3, smem = 8 * (kS * kChunk * 128 + kChunk * 32);
        if ((e = staged_grid(combine_encode_staged<false, kS>, smem, nchunks, &g)) != cudaSuccess) return e;
        combine_encode_staged<false, kS><<<g, 256, smem, st>>>(in, groups, signs, codes, e8m0);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k,
                                  int64_t cols, uint32_t signs, void* out, int out_bf16, cudaStream_t st) {
    const int64_t gpr = cols / 32;
    constexpr int kS = 3;
    const int64_t smem64 = 8 * (kS * k * (1024 + 32) + kChunk * (out_bf16 ? 64 : 128));
    if (gpr % kChunk == 0 && ((uintptr_t)e8m0 & 3) == 0 && smem64 <= 227 * 1024) {
        const int smem = (int)smem64;
        const int64_t nchunks = tokens * gpr / kChunk;
        unsigned g = 0;
        cudaError_t e;
        if (out_bf16) {
            if ((e = staged_grid(combine_decode_staged<true, kS>, smem, nchunks, &g)) != cudaSuccess) return e;
            combine_decode_staged<true, kS><<<g, 256, smem, st>>>(codes, e8m0, tokens, (int)k, gpr, signs, out);
        } else {
            if ((e = staged_grid(combine_decode_staged<false, kS>, smem, nchunks, &g)) != cudaSuccess) return e;
            combine_decode_staged<false, kS><<<g, 256, smem, st>>>(codes, e8m0, tokens, (int)k, gpr, signs, out);
        }
        return cudaGetLastError();
    }
    const unsigned g = combine_grid(tokens * gpr);
    if (out_bf16)
        combine_decode_kernel<true><<<g, 256, 0, st>>>(codes, e8m0, tokens, k, gpr, signs, out);
    else
        combine_decode_kernel<false><<<g, 256, 0, st>>>(codes, e8m0, tokens, k, gpr, signs, out);
    return cudaGetLastError();
}

}  // namespace fp4q
