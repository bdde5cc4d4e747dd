// fp4q_internal.h — launchers shared between the kernel translation units and the C ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fp4q {

int num_sms();            // SM count of the current device (cached per device)
int check_device();       // FP4Q_OK on a compute-capability 10.x device (cached per device)
bool use_hw_e2m1();       // convert E2M1 with the hardware cvt (shown equal to the ALU rule)

cudaError_t launch_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                        int64_t batch_stride, float* out, cudaStream_t st);
cudaError_t launch_quantize_1d(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                               const float* amax, uint8_t* codes, uint8_t* scales, float* s_dec,
                               cudaStream_t st);
cudaError_t launch_quantize_1d_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int four_six,
                                    uint8_t* codes, uint8_t* scales, float* s_dec_rows, cudaStream_t st);
void rows_shape(int64_t cols, int& W, int& hold);   // warps per row, blocks per thread
cudaError_t launch_quantize_mxfp4(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int rht, uint32_t signs,
                                  uint8_t* codes, uint8_t* e8m0, cudaStream_t st);
cudaError_t launch_quantize_2d(const uint16_t* w, int64_t rows, int64_t cols, int64_t ld,
                               int64_t batch, int64_t batch_stride, const float* amax,
                               uint8_t* codes, uint8_t* tile_scales, float* s_dec,
                               cudaStream_t st);

struct RequantArgs {
    int in_kind;                 // 0 bf16, 1 NVFP4 1D, 2 NVFP4 2D, 3 NVFP4 1D with per-row s_dec
    const void* in;
    const uint8_t* in_scales;
    const float* in_s_dec;       // one float, or [rows] for kind 3
    int64_t rows, cols;
    int transpose, rht;
    uint32_t rht_signs;
    int rounding;                // 0 RNE, 1 SR
    uint64_t seed;
    uint32_t tag;
    uint8_t* out_e4m3;
    uint8_t* out_e8m0;
    // bf16 input only: a second, rowwise output from the same read (no transform, tag2)
    uint8_t* out2_e4m3 = nullptr;
    uint8_t* out2_e8m0 = nullptr;
    uint32_t tag2 = 0;
};
cudaError_t launch_requant(const RequantArgs& a, cudaStream_t st);
cudaError_t launch_combine_encode(const void* in, int in_bf16, int64_t rows, int64_t cols, uint32_t signs,
                                  uint8_t* codes, uint8_t* e8m0, cudaStream_t st);
cudaError_t launch_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k,
                                  int64_t cols, uint32_t signs, void* out, int out_bf16, cudaStream_t st);
cudaError_t launch_rht16(const void* in, int in_is_bf16, float* out, int64_t rows, int64_t cols,
                         uint32_t signs, cudaStream_t st);

struct GemmArgs {
    int kind;                    // 0 NVFP4, 1 MXFP8, 2 MXFP4 (E8M0 scales per 32; K % 2048 == 0)
    const uint8_t* a;
    const uint8_t* a_scales;
    const float* a_s_dec;        // NVFP4 only: one float, or [M] when a_sdec_rows
    const uint8_t* b;
    const uint8_t* b_scales;
    int b_scale_kind;            // NVFP4: 1 = 1D, 2 = 16x16 tiles
    const float* b_s_dec;        // NVFP4 only, [groups]
    void* d;
    int d_bf16;
    int64_t M, N, K;
    int groups;
    const int64_t* group_offsets;   // host, groups + 1 (NULL when groups == 1)
    // epilogue: 0 plain; 1 GELU (bf16): d = h, d2 = GELU(h), amax_out = max|d2|;
    // 2 GELU backward (bf16): d = bf16(d_bf16 * GELU'(aux)), aux = the layer's pre-activation h;
    // 3 combine encode (d_bf16 = 0): RHT32 + S2F6 of each row's groups of 32
    int epi = 0;
    void* d2 = nullptr;
    const uint16_t* aux = nullptr;
    float* amax_out = nullptr;   // epi 1; may be NULL
    uint32_t rht32_signs = 0;    // epi 3: combine encode (d = S2F6 bytes, d2 = E8M0 per 32), fp32 path
    int a_sdec_rows = 0;         // NVFP4: A carries one outer scale per row
    // failure-detection test (CTA-pair kernel only): every mbarrier wait gives up after
    // wait_limit_ns (0: the default 1.5 s), and with no_copies the producers issue no copies,
    // so the waits run out, the kernel raises the device error word and returns
    int64_t wait_limit_ns = 0;
    int no_copies = 0;
};
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st);
int read_and_clear_device_error(cudaStream_t st, int* flag);

}  // namespace fp4q
