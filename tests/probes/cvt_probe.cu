// cvt_probe.cu — test-only kernels that exercise device building blocks of the library in
// isolation: the E2M1 / E4M3 encoders against the hardware conversion instructions, the
// hardware stochastic rounding and the f16x2 dequantization path, and
// the Philox4x32-10 generator against cuRAND's implementation of the same published
// generator. Every kernel is one thread per element with a bounds check; nothing waits.
#include <cstdint>
#include <curand_philox4x32_x.h>
#include "../../mxfp8_precision_numerics_gb300/csrc/fp4q_common.cuh"

namespace {

__global__ void e2m1_kernel(const float* in, uint8_t* alu, uint8_t* hw_lo, uint8_t* hw_hi, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = in[i];
    alu[i] = (uint8_t)fp4q::e2m1_rne_alu(v);
    hw_lo[i] = (uint8_t)fp4q::e2m1x2_cvt_rn(v, 0.0f);     // whole byte: v requested in the low nibble
    hw_hi[i] = (uint8_t)fp4q::e2m1x2_cvt_rn(0.0f, v);     // whole byte: v requested in the high nibble
}

// hw_first: v as the first source operand, hw_second: v as the second (16-bit results)
__global__ void e4m3_kernel(const float* in, uint8_t* alu, uint16_t* hw_first, uint16_t* hw_second,
                            int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = in[i];
    alu[i] = (uint8_t)fp4q::e4m3_rne_sat(v);
    unsigned short s1, s2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s1) : "f"(v), "f"(0.0f));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s2) : "f"(0.0f), "f"(v));
    hw_first[i] = s1;
    hw_second[i] = s2;
}

__global__ void e4m3_sr_kernel(const float* in, const uint32_t* r16, uint8_t* out, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    out[i] = (uint8_t)fp4q::e4m3_sr(in[i], r16[i]);
}

// Hardware stochastic rounding of (even, odd) pairs with one random word per pair: the
// whole 32-bit result is returned so that the test also sees the unused bytes.
__global__ void e4m3x2_sr_hw_kernel(const float* in, const uint32_t* rbits, uint32_t* out, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    out[i] = fp4q::e4m3x2_sr_hw(in[2 * i], in[2 * i + 1], rbits[i]);
}

// Dequantization of eight packed E2M1 codes with one E4M3 block scale and an fp32 tensor
// scale, through the f16x2 conversion path (f16) and the plain fp32 decode (ref).
__global__ void dequant8_kernel(const uint32_t* words, const uint8_t* scales, float s_dec, float* f16,
                                float* ref, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint32_t w = words[i], sc = scales[i];
    fp4q::dequant8_f16(w, fp4q::e4m3_to_f16x2_dup(sc), s_dec, f16 + 8 * i);
    const float scf = fp4q::e4m3_to_f32(sc);
    for (int j = 0; j < 8; ++j)
        ref[8 * i + j] = __fmul_rn(__fmul_rn(fp4q::e2m1_to_f32((w >> (4 * j)) & 15u), scf), s_dec);
}

__global__ void philox_kernel(const uint32_t* ctr, const uint32_t* key, uint32_t* mine,
                              uint32_t* ref, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    uint2 k = make_uint2(key[2 * i], key[2 * i + 1]);
    uint4 a = fp4q::philox4x32_10(c, k.x, k.y);
    uint4 b = curand_Philox4x32_10(c, k);
    mine[4 * i] = a.x; mine[4 * i + 1] = a.y; mine[4 * i + 2] = a.z; mine[4 * i + 3] = a.w;
    ref[4 * i] = b.x; ref[4 * i + 1] = b.y; ref[4 * i + 2] = b.z; ref[4 * i + 3] = b.w;
}

__global__ void mx_exp_kernel(const float* amax, int* e, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    e[i] = fp4q::mx_exponent(amax[i]);
}

inline unsigned blocks(int n) { return (unsigned)((n + 255) / 256); }

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int probe_e2m1(const float* in, uint8_t* alu, uint8_t* hw_lo,
                                                       uint8_t* hw_hi, int n, cudaStream_t st) {
    if (n <= 0) return 0;
    e2m1_kernel<<<blocks(n), 256, 0, st>>>(in, alu, hw_lo, hw_hi, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_e4m3(const float* in, uint8_t* alu, uint16_t* hw_first,
                                                       uint16_t* hw_second, int n, cudaStream_t st) {
    if (n <= 0) return 0;
    e4m3_kernel<<<blocks(n), 256, 0, st>>>(in, alu, hw_first, hw_second, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_e4m3_sr(const float* in, const uint32_t* r16, uint8_t* out,
                                                          int n, cudaStream_t st) {
    if (n <= 0) return 0;
    e4m3_sr_kernel<<<blocks(n), 256, 0, st>>>(in, r16, out, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_e4m3x2_sr_hw(const float* in, const uint32_t* rbits,
                                                              uint32_t* out, int n, cudaStream_t st) {
    if (n <= 0) return 0;
    e4m3x2_sr_hw_kernel<<<blocks(n), 256, 0, st>>>(in, rbits, out, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_dequant8(const uint32_t* words, const uint8_t* scales,
                                                          float s_dec, float* f16, float* ref, int n,
                                                          cudaStream_t st) {
    if (n <= 0) return 0;
    dequant8_kernel<<<blocks(n), 256, 0, st>>>(words, scales, s_dec, f16, ref, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_philox(const uint32_t* ctr, const uint32_t* key,
                                                         uint32_t* mine, uint32_t* ref, int n,
                                                         cudaStream_t st) {
    if (n <= 0) return 0;
    philox_kernel<<<blocks(n), 256, 0, st>>>(ctr, key, mine, ref, n);
    return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int probe_mx_exponent(const float* amax, int* e, int n,
                                                              cudaStream_t st) {
    if (n <= 0) return 0;
    mx_exp_kernel<<<blocks(n), 256, 0, st>>>(amax, e, n);
    return (int)cudaGetLastError();
}

}  // extern "C"
