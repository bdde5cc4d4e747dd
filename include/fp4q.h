/*
 * fp4q.h — C ABI of libfp4q.so: the hot path of the NVFP4 linear layer on one GB300.
 *
 * Forward: NVFP4 quantize of activations (1x16 blocks) and weights (16x16 tiles), then a
 * block-scaled NVFP4 x NVFP4 GEMM with FP32 accumulation. Backward: dequantize, transpose
 * and re-quantize to MXFP8 with stochastic rounding, an optional 16-point random Hadamard
 * transform on the wgrad operands, then MXFP8 dgrad / wgrad GEMMs.
 *
 * Sources (web pages, by title and section):
 *   [NV]  "Pretraining Large Language Models with NVFP4" (arXiv 2509.25149), summary page:
 *         "NVFP4 Format and Quantization Procedure" steps 1-5; "Random Hadamard Transforms";
 *         "Two-Dimensional Weight Scaling and the Chain Rule Problem";
 *         "Stochastic Rounding for Unbiased Gradients".
 *   [VZ]  "End-to-End 4-Bit Training" rebuilt on one B200 (4bit.vizuara.ai), §5-§13.
 *   [TML] "End-to-End 4-Bit Training" (Thinking Machines), "基于随机舍入的重量化".
 *   [AC]  "FP4 Training on Blackwell" (aicassindra.com), "The scaling math, worked".
 *
 * Conventions shared by every entry point
 *   - All tensors are row-major. bf16 inputs are 16-bit IEEE bfloat16.
 *   - Pointers are device pointers unless stated otherwise. The caller owns and allocates
 *     every buffer, including the small workspaces; the library allocates nothing and keeps
 *     no state between calls other than a device-side error word (fp4q_device_status).
 *   - Work is enqueued asynchronously on `stream` (NULL = the legacy default stream). Scalars
 *     (amax, s_dec) stay on the device; no call synchronizes the host.
 *   - Arguments are validated on the host before any launch. A failed check returns a
 *     status and launches nothing. A launch error maps to FP4Q_ERR_CUDA.
 *   - Packed NVFP4 codes: E2M1, two per byte, element 2j in the low nibble, 2j+1 in the high
 *     nibble; a row of `cols` values takes cols/2 bytes. NVFP4 block scales: one E4M3 byte
 *     per block, row-major. MXFP8: one E4M3 byte per value plus one E8M0 byte per 32
 *     consecutive values of a row (value = e4m3 * 2^(e8m0 - 127)).
 *   - Non-finite inputs (inf, NaN) are outside the method; their outputs are unspecified.
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP4Q_API __attribute__((visibility("default")))
#else
#define FP4Q_API
#endif

/* A CUDA stream handle (the same object as cudaStream_t). */
typedef struct CUstream_st* fp4q_stream_t;

enum fp4q_status {
    FP4Q_OK = 0,
    FP4Q_ERR_NULL = 1,        /* a required pointer is NULL                               */
    FP4Q_ERR_ALIGN = 2,       /* a pointer or leading dimension breaks the 16-byte rule    */
    FP4Q_ERR_SHAPE = 3,       /* a size is zero, negative or not a required multiple       */
    FP4Q_ERR_ARG = 4,         /* an enum or flag argument is out of range                  */
    FP4Q_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed                      */
    FP4Q_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up (fp4q_device_status)  */
    FP4Q_ERR_UNSUPPORTED = 7  /* the current device is not sm_103 / sm_100 class          */
};

enum fp4q_in_kind { FP4Q_IN_BF16 = 0, FP4Q_IN_NVFP4_1D = 1, FP4Q_IN_NVFP4_2D = 2,
                    FP4Q_IN_NVFP4_1D_ROWS = 3 };
enum fp4q_rounding { FP4Q_RNE = 0, FP4Q_SR = 1 };
enum fp4q_dtype { FP4Q_F32 = 0, FP4Q_BF16 = 1 };
enum fp4q_scale_kind { FP4Q_SCALE_1D = 1, FP4Q_SCALE_2D = 2 };

/* Human-readable name of a status code (static string, never NULL). */
FP4Q_API const char* fp4q_status_str(int status);

/* ABI version of this header (major * 100 + minor). */
FP4Q_API int fp4q_version(void);

/*
 * fp4q_quantize_1d — NVFP4 quantize with 1x16 blocks along each row.
 * [NV] "NVFP4 Format and Quantization Procedure", steps 1-4; [VZ] §5-6.
 *   amax   = max |x| over the tensor                      (step 1; the extra HBM pass)
 *   s_enc  = 2688 / amax (fp32), s_dec = 1 / s_enc;  amax == 0 -> s_enc = s_dec = 1
 *   per block b of 16: sb = E4M3_RNE((amax_b / 6) * s_enc), raised to 0x01 if it is 0
 *                      s_enc_b = 1 / (fp32(sb) * s_dec)
 *                      code_i = E2M1_RNE(x_i * s_enc_b)    (ties to even, saturating)
 *   x_bf16    [rows][ld] bf16, 16-byte aligned, ld % 8 == 0, ld >= cols
 *   amax_in   device float or NULL. If given, it is used as the tensor amax (for example an
 *             amax agreed across shards) and amax_ws may be NULL.
 *   amax_ws   device float workspace (4 bytes) that receives the computed amax; required when
 *             amax_in is NULL. It is overwritten.
 *   codes     [rows][cols/2] bytes, 16-byte aligned; scales [rows][cols/16] E4M3 bytes
 *   s_dec_out device float: the per-tensor decode scale s_dec.
 *   rows >= 1, cols >= 16, cols % 16 == 0.
 */
FP4Q_API int fp4q_quantize_1d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                     const float* amax_in, float* amax_ws,
                     uint8_t* codes, uint8_t* scales, float* s_dec_out, fp4q_stream_t stream);

/*
 * fp4q_quantize_1d_rows — NVFP4 quantize with 1x16 blocks along each row, one FP32 outer scale
 * per row (per token) and, if four_six, the Four Over Six block-scale choice: the activation
 * quantizer of 4bit.vizuara.ai §10 (QLinearFn: outer="row", four_six=True) and of the
 * Thinking Machines recipe ("End-to-End 4-Bit Training", 方案细节). One pass over x; no
 * amax kernel and no workspace.
 *   per row r: amax_r = max |x[r, :]|; s_enc = 2688 / amax_r, s_dec = 1 / s_enc (fp32;
 *              amax_r == 0 -> 1 and 1); s_dec_rows[r] = s_dec
 *   per block, candidate c = 6 (and c = 4 when four_six):
 *              sb_c = E4M3_RNE((amax_b / c) * s_enc), saturating, raised to 0x01 if 0;
 *              s_enc_b = 1 / (fp32(sb_c) * s_dec); y_i = x_i * s_enc_b; code_i = E2M1_RNE(y_i)
 *              E_c = (sum_i (y_i - q_i)^2) * fp32(sb_c)^2, q_i = E2M1 value of code_i; the
 *              squares are summed with fused multiply-adds in two chains (even positions,
 *              odd positions), each in index order, and the chains are added
 *              the block keeps candidate 4 iff E_4 < E_6 (the choice lives in the scale byte)
 *   x_bf16      [rows][ld] bf16, 16-byte aligned, ld % 8 == 0, ld >= cols
 *   four_six    0 or 1
 *   codes       [rows][cols/2] bytes, 16-byte aligned; scales [rows][cols/16] E4M3 bytes
 *   s_dec_rows  device float[rows]
 *   rows >= 1, cols >= 16, cols % 16 == 0.
 * Decode: x^[r, k] = E2M1(code) * E4M3(scale) * s_dec_rows[r]; fp4q_gemm_nvfp4_rows and the
 * requantize input kind FP4Q_IN_NVFP4_1D_ROWS take this form.
 */
FP4Q_API int fp4q_quantize_1d_rows(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                     int four_six, uint8_t* codes, uint8_t* scales, float* s_dec_rows,
                     fp4q_stream_t stream);

/*
 * fp4q_quantize_2d — NVFP4 quantize of a weight with one E4M3 scale per 16x16 tile, so the
 * row-wise and column-wise views share scales. [NV] "Two-Dimensional Weight Scaling and the
 * Chain Rule Problem"; [VZ] §8. Same arithmetic as fp4q_quantize_1d with amax_b taken over
 * the 256 values of a tile. `batch` independent tensors (e.g. MoE experts), each with its
 * own amax and s_dec, sit `batch_stride` elements apart.
 *   w_bf16      [batch][rows][ld] bf16, 16-byte aligned, ld % 8 == 0, batch_stride % 8 == 0
 *   amax_in     device float[batch] or NULL; amax_ws device float[batch] (required if
 *               amax_in is NULL)
 *   codes       [batch][rows][cols/2];  tile_scales [batch][rows/16][cols/16]
 *   s_dec_out   device float[batch]
 *   rows % 16 == 0, cols % 16 == 0, batch >= 1.
 */
FP4Q_API int fp4q_quantize_2d(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                     int64_t batch, int64_t batch_stride,
                     const float* amax_in, float* amax_ws,
                     uint8_t* codes, uint8_t* tile_scales, float* s_dec_out,
                     fp4q_stream_t stream);

/*
 * fp4q_quantize_2d_noalloc — fp4q_quantize_2d for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point: it is an interface convenience.
 * Some callers cannot call cudaMalloc: a plugin whose host framework owns every device buffer
 * and offers no workspace, or a latency-critical caller that must avoid cudaMalloc because it
 * can synchronize the device. Here the per-tensor amax workspace is a fixed array inside the
 * library (FP4Q_NOALLOC_MAX_BATCH floats, 4 KiB per device, kept until the process exits); the
 * caller passes only inputs and outputs, with the same meaning, layout and results as
 * fp4q_quantize_2d computing its own amax.
 *   batch > FP4Q_NOALLOC_MAX_BATCH is rejected with FP4Q_ERR_SHAPE before any launch.
 *   The first call on a device looks up the array's device address (once per device, with
 *   that device current, and again after the device's context changes, e.g. after a
 *   cudaDeviceReset); make that first call before any stream capture.
 *   Every call on a device shares the array: calls whose work may overlap on the GPU (two
 *   streams without ordering between them) race on it. Calls ordered on one stream are safe;
 *   each call clears the part it uses before accumulating the amax.
 *   The library allocates nothing for this call.
 */
#define FP4Q_NOALLOC_MAX_BATCH 1024
FP4Q_API int fp4q_quantize_2d_noalloc(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                                      int64_t batch, int64_t batch_stride,
                                      uint8_t* codes, uint8_t* tile_scales, float* s_dec_out,
                                      fp4q_stream_t stream);

/*
 * fp4q_requant_t_mxfp8_sr — dequantize, optionally transpose, optionally apply the 16-point
 * random Hadamard transform, and quantize to MXFP8 with stochastic rounding.
 * [VZ] §9-10 ("each saved tensor is dequantized, transposed and re-quantized to MXFP8 with
 * SR"); [TML] "基于随机舍入的重量化"; [NV] "Random Hadamard Transforms" (wgrad operands);
 * [AC] "The scaling math, worked" (power-of-two ceiling scale).
 *   in_kind   FP4Q_IN_BF16: in = bf16 [rows][cols]; in_scales, in_s_dec unused (may be NULL)
 *             FP4Q_IN_NVFP4_1D: in = codes [rows][cols/2], in_scales [rows][cols/16],
 *                               in_s_dec = device float
 *             FP4Q_IN_NVFP4_2D: in = codes [rows][cols/2], in_scales [rows/16][cols/16]
 *             FP4Q_IN_NVFP4_1D_ROWS: as FP4Q_IN_NVFP4_1D with in_s_dec = device float[rows],
 *                               one outer scale per input row (fp4q_quantize_1d_rows)
 *   dequantized value (fp32) = (E2M1(code) * E4M3(scale)) * s_dec (of the input row for
 *             FP4Q_IN_NVFP4_1D_ROWS)
 *   transpose 0: output [rows][cols]; 1: output [cols][rows]. MXFP8 blocks of 32 and the
 *             Hadamard groups of 16 run along the OUTPUT's contiguous dimension.
 *   rht       0 / 1. The transform on each group of 16: y = (1/4) H16 (s o x), Sylvester H16,
 *             bit i of rht_signs set -> s_i = -1; evaluated as butterflies at distances
 *             1, 2, 4, 8 in fp32, then the exact multiply by 1/4.
 *   per block of 32: e = the smallest integer with amax <= 448 * 2^e, clamped to [-127, 127];
 *             out_e8m0 = e + 127; element = E4M3(x * 2^-e) rounded by `rounding`.
 *   rounding  FP4Q_SR: floor(t/step + U) on the local E4M3 grid, U = R/2^16, where R is the
 *             16-bit slice for the element's linear output index i of Philox4x32-10 with
 *             key (seed lo32, seed hi32) and counter (i>>3 lo32, i>>3 hi32, tensor_tag, 0):
 *             word (i>>1)&3, low half for even i, high half for odd i.
 *             FP4Q_RNE: round to nearest, ties to even.
 *   out_e4m3  [out_rows][out_cols] bytes; out_e8m0 [out_rows][out_cols/32] bytes
 *   rows % 32 == 0 and cols % 32 == 0; for FP4Q_IN_NVFP4_2D also rows % 16 == 0.
 *   in is 16-byte aligned; out_e4m3 is 16-byte aligned.
 */
FP4Q_API int fp4q_requant_t_mxfp8_sr(int in_kind, const void* in, const uint8_t* in_scales,
                            const float* in_s_dec, int64_t rows, int64_t cols,
                            int transpose, int rht, uint32_t rht_signs,
                            int rounding, uint64_t seed, uint32_t tensor_tag,
                            uint8_t* out_e4m3, uint8_t* out_e8m0, fp4q_stream_t stream);

/*
 * fp4q_requant_bf16_dual — the output gradient's two MXFP8 quantizations from one read of it:
 * the rowwise one for dgrad and the transposed one (optionally with the 16-point transform) for
 * wgrad ([VZ] §10: "the output gradient is quantized to MXFP8 twice, as it is and transposed";
 * [NV] "Random Hadamard Transforms" for the wgrad operand). The results are exactly those of
 *   fp4q_requant_t_mxfp8_sr(FP4Q_IN_BF16, in, ..., transpose = 0, rht = 0, ..., tag_rows, rows_*)
 *   fp4q_requant_t_mxfp8_sr(FP4Q_IN_BF16, in, ..., transpose = 1, rht, ..., tag_t, t_*)
 * with the same rounding and seed (each output keeps its own counter stream, tagged).
 *   in bf16 [rows][cols]; rows_e4m3 [rows][cols], rows_e8m0 [rows][cols/32];
 *   t_e4m3 [cols][rows], t_e8m0 [cols][rows/32].
 *   rows, cols multiples of 32; in, rows_e4m3, t_e4m3 16-byte aligned; errors as
 *   fp4q_requant_t_mxfp8_sr.
 */
FP4Q_API int fp4q_requant_bf16_dual(const void* in, int64_t rows, int64_t cols, int rht, uint32_t rht_signs,
                    int rounding, uint64_t seed, uint32_t tag_rows, uint32_t tag_t,
                    uint8_t* rows_e4m3, uint8_t* rows_e8m0, uint8_t* t_e4m3, uint8_t* t_e8m0,
                    fp4q_stream_t stream);

/*
 * fp4q_rht16 — the 16-point random Hadamard transform on its own, along rows.
 * [NV] "Random Hadamard Transforms"; [AC] "Hadamard rotations". Same arithmetic and order
 * as the transform inside fp4q_requant_t_mxfp8_sr.
 *   in        [rows][cols], in_dtype FP4Q_F32 or FP4Q_BF16, 16-byte aligned
 *   out       [rows][cols] fp32, 16-byte aligned (may alias `in` when in_dtype == FP4Q_F32)
 *   cols % 16 == 0.
 */
FP4Q_API int fp4q_rht16(const void* in, int in_dtype, float* out, int64_t rows, int64_t cols,
               uint32_t signs, fp4q_stream_t stream);

/*
 * fp4q_gemm_nvfp4 — block-scaled NVFP4 x NVFP4 GEMM, D = A . B^T, FP32 accumulation on the
 * tcgen05 tensor cores. [NV] "NVFP4 Format and Quantization Procedure", step 5:
 *   D[m,n] = s_dec_a * s_dec_b * sum_blocks sa[m,blk] * sb[n,blk] * sum_{k in blk} a_k b_k
 *   a, a_scales, a_s_dec    codes [M][K/2], E4M3 [M][K/16] (1D), device float
 *   b, b_scales, b_s_dec    codes [groups][N][K/2]; scales [groups][N][K/16] (b_scale_kind
 *                           FP4Q_SCALE_1D) or [groups][N/16][K/16] (FP4Q_SCALE_2D, each tile
 *                           scale serves its 16 rows); b_s_dec device float[groups]
 *   d, d_dtype              [M][N] FP4Q_F32 or FP4Q_BF16 (round to nearest even)
 *   groups, group_row_offsets_host
 *                           groups == 1: offsets may be NULL. groups > 1 (grouped GEMM, MoE
 *                           experts): HOST int64 array of groups+1 ascending row offsets into
 *                           A and D with offsets[0] = 0 and offsets[groups] = M; rows of group
 *                           g multiply B[g]. groups <= 64.
 *   M >= 1, N % 16 == 0, K % 256 == 0 (whole 256-value pipeline stages); a, b, a_scales,
 *   b_scales and d 16-byte aligned.
 */
FP4Q_API int fp4q_gemm_nvfp4(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, void* d, int d_dtype,
                    int64_t M, int64_t N, int64_t K,
                    int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream);

/*
 * fp4q_gemm_nvfp4_rows — fp4q_gemm_nvfp4 with one outer scale per row of A, the activation form
 * of 4bit.vizuara.ai §10 (per-token outer scale; fp4q_quantize_1d_rows produces it):
 *   D[m,n] = s_dec_a[m] * s_dec_b[g] * sum_blocks sa[m,blk] * sb[n,blk] * sum_{k in blk} a_k b_k
 *   a_s_dec_rows  device float[M]; every other argument as fp4q_gemm_nvfp4.
 */
FP4Q_API int fp4q_gemm_nvfp4_rows(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec_rows,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, void* d, int d_dtype,
                    int64_t M, int64_t N, int64_t K,
                    int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream);

/*
 * fp4q_gemm_mxfp8 — block-scaled MXFP8 x MXFP8 GEMM, D = A . B^T, FP32 accumulation on the
 * tcgen05 tensor cores (the dgrad and wgrad GEMMs of the backward pass). [VZ] §8 and §10:
 * dx = g . w_q sums over N, dw = g^T . x_q sums over tokens; both operands carry their
 * E8M0 block scales along the contraction dimension.
 *   D[m,n] = sum_blk 2^(ea[m,blk]-127) * 2^(eb[n,blk]-127) * sum_{k in blk} a_k b_k
 *   a, a_scales   E4M3 [M][K], E8M0 [M][K/32];  b, b_scales  E4M3 [N][K], E8M0 [N][K/32]
 *   d, d_dtype    [M][N] FP4Q_F32 or FP4Q_BF16
 *   M >= 1, N % 16 == 0, K % 128 == 0 (whole 128-value pipeline stages); a, b, d 16-byte
 *   aligned; a_scales and b_scales 4-byte aligned.
 */
FP4Q_API int fp4q_gemm_mxfp8(const uint8_t* a, const uint8_t* a_scales,
                    const uint8_t* b, const uint8_t* b_scales,
                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                    fp4q_stream_t stream);

/*
 * fp4q_gemm_nvfp4_gelu — fp4q_gemm_nvfp4 (groups == 1, bf16 output) with the MLP's activation
 * fused into the epilogue: the first linear layer of a GPT MLP block, whose output feeds GELU
 * and then the second layer's 1D NVFP4 quantization ([VZ] §13-14 pairs GELU with the quantize
 * of its output). GELU is the exact-erf form x * Phi(x) evaluated in fp32 on the bf16 h.
 *   h_out      [M][N] bf16 = the GEMM output (round to nearest even), as fp4q_gemm_nvfp4 writes it
 *   act_out    [M][N] bf16 = GELU(h_out), round to nearest even
 *   act_amax   device float: max |act_out| over the tensor, bit-exact, ready as the `amax_in`
 *              of fp4q_quantize_1d(act_out) (which then skips its own amax pass)
 *   Other arguments, shapes and alignment as fp4q_gemm_nvfp4 with groups == 1; h_out and
 *   act_out 16-byte aligned.
 */
FP4Q_API int fp4q_gemm_nvfp4_gelu(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, void* h_out, void* act_out, float* act_amax,
                    int64_t M, int64_t N, int64_t K, fp4q_stream_t stream);

/*
 * fp4q_gemm_nvfp4_gelu_rows — fp4q_gemm_nvfp4_gelu with one outer scale per row of A
 * (a_s_dec_rows, device float[M]). act_amax may be NULL (a per-row quantizer of act_out needs
 * no tensor amax); if given it receives max |act_out| as in fp4q_gemm_nvfp4_gelu.
 */
FP4Q_API int fp4q_gemm_nvfp4_gelu_rows(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec_rows,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, void* h_out, void* act_out, float* act_amax,
                    int64_t M, int64_t N, int64_t K, fp4q_stream_t stream);

/*
 * fp4q_gemm_mxfp8_dgelu — fp4q_gemm_mxfp8 (bf16 output) with the activation's backward fused
 * into the epilogue: the dgrad GEMM of the MLP's second layer produces dL/d(act); the
 * epilogue rounds it to bf16 and multiplies by GELU'(h) = Phi(h) + h * phi(h) in fp32, giving
 * dL/dh for the first layer's backward.
 *   h          [M][N] bf16, the first layer's pre-activation (h_out of fp4q_gemm_nvfp4_gelu)
 *   dh_out     [M][N] bf16 = bf16( bf16(A . B^T) * GELU'(h) ), round to nearest even
 *   Other arguments, shapes and alignment as fp4q_gemm_mxfp8; h and dh_out 16-byte aligned.
 */
FP4Q_API int fp4q_gemm_mxfp8_dgelu(const uint8_t* a, const uint8_t* a_scales,
                    const uint8_t* b, const uint8_t* b_scales, const void* h, void* dh_out,
                    int64_t M, int64_t N, int64_t K, fp4q_stream_t stream);

/*
 * fp4q_quantize_mxfp4 — MXFP4, the Open Compute microscaling format the NVFP4 paper compares
 * against: E2M1 codes with one E8M0 scale per 32 values of a row. [AC] "The scaling math,
 * worked" (scale = 2^ceil(log2(amax / 6))); [NV] Section 5 and App. B.4.
 *   per group of 32 (optionally rotated first: rht = 1 applies the RHT32 of the combine format
 *   below, the 32-point transform the paper pairs with MXFP4): e = the smallest integer with
 *   amax <= 6 * 2^e, clamped to [-127, 127]; e8m0 = e + 127; code_i = E2M1_RNE(x_i * 2^-e)
 *   x_bf16    [rows][ld] bf16, 16-byte aligned, ld % 8 == 0
 *   codes     [rows][cols/2] (element 2j low nibble), 16-byte aligned; e8m0 [rows][cols/32]
 *   rows >= 1, cols % 32 == 0.
 */
FP4Q_API int fp4q_quantize_mxfp4(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, int rht,
                    uint32_t rht_signs, uint8_t* codes, uint8_t* e8m0, fp4q_stream_t stream);

/*
 * fp4q_gemm_mxfp4 — block-scaled MXFP4 x MXFP4 GEMM, D = A . B^T, FP32 accumulation on the
 * tcgen05 tensor cores (block-scaled E2M1 MMA with UE8M0 scales, two per row and MMA):
 *   D[m,n] = sum_blk 2^(ea[m,blk]-127) * 2^(eb[n,blk]-127) * sum_{k in blk} a_k b_k
 *   a, a_e8m0   codes [M][K/2], E8M0 [M][K/32];  b, b_e8m0  codes [N][K/2], E8M0 [N][K/32]
 *   d, d_dtype  [M][N] FP4Q_F32 or FP4Q_BF16
 *   M >= 1, N % 16 == 0, K % 2048 == 0 (the kernel stages the scales of 2048 values of K at a
 *   time); all pointers 16-byte aligned.
 */
FP4Q_API int fp4q_gemm_mxfp4(const uint8_t* a, const uint8_t* a_e8m0, const uint8_t* b, const uint8_t* b_e8m0,
                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K, fp4q_stream_t stream);

/*
 * The MoE combine wire format: RHT32 + block-scaled S2F6 ([VZ] §11, "Combine is harder";
 * [TML] 合并阶段). A layer output is rotated in groups of 32 consecutive values of a row and
 * sent as S2F6 (8.25 bits per value); the receiver sums the dequantized arrivals of a token
 * and rotates the sum back.
 *   rotation  y = c * H32 (s o x): bit i of rht_signs set -> s_i = -1; Sylvester H32 evaluated
 *             as butterflies at distances 1, 2, 4, 8, 16 in fp32; c = RN(1/sqrt 32) applied to
 *             each value once. Inverse: butterflies, c, then the signs.
 *   S2F6      e = the smallest integer with max|y| <= (127/64) 2^e over the group, clamped to
 *             [-127, 127]; E8M0 byte e + 127; code q = round-half-even(y 2^(6-e)) clamped to
 *             [-128, 127], stored as a two's-complement byte; value q 2^(e-6).
 */

/*
 * fp4q_combine_encode — rotate and quantize a [rows][cols] tensor (groups of 32 along rows).
 *   x          fp32 or bf16 (x_dtype FP4Q_F32 / FP4Q_BF16) [rows][cols], 16-byte aligned
 *   codes      [rows][cols] S2F6 bytes, 16-byte aligned; e8m0 [rows][cols/32]
 *   rows >= 1, cols % 32 == 0.
 */
FP4Q_API int fp4q_combine_encode(const void* x, int x_dtype, int64_t rows, int64_t cols, uint32_t rht_signs,
                    uint8_t* codes, uint8_t* e8m0, fp4q_stream_t stream);

/*
 * fp4q_combine_decode — sum each token's k arrivals and rotate the sum back.
 *   codes, e8m0  [tokens * k][cols] and [tokens * k][cols/32]: token t's arrivals are rows
 *                t*k .. t*k+k-1, summed in fp32 in that order (exact dequantized values)
 *   out          [tokens][cols] fp32 or bf16 (out_dtype; bf16 = round to nearest even of the
 *                fp32 result), 16-byte aligned; codes 16-byte aligned
 *   tokens >= 1, k >= 1, cols % 32 == 0.
 */
FP4Q_API int fp4q_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k,
                    int64_t cols, uint32_t rht_signs, void* out, int out_dtype, fp4q_stream_t stream);

/*
 * fp4q_gemm_nvfp4_combine — fp4q_gemm_nvfp4 (grouped or not) whose epilogue rotates each row's
 * groups of 32 output values and writes them in the combine wire format instead of a float
 * output ([VZ] §11: rotation and conversion at the very end of the GEMM kernel). The values
 * encoded are the fp32 outputs fp4q_gemm_nvfp4 would store (accumulator x s_dec_a x s_dec_b).
 *   codes_out  [M][N] S2F6 bytes, 16-byte aligned; e8m0_out [M][N/32]
 *   N % 32 == 0; every other argument as fp4q_gemm_nvfp4.
 */
FP4Q_API int fp4q_gemm_nvfp4_combine(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, uint32_t rht_signs, uint8_t* codes_out, uint8_t* e8m0_out,
                    int64_t M, int64_t N, int64_t K,
                    int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream);

/*
 * fp4q_device_status — synchronizes `stream`, then reads and clears the library's device-side
 * error word. Returns FP4Q_ERR_TIMEOUT if a kernel's bounded wait (a GEMM pipeline barrier)
 * gave up since the last call, FP4Q_ERR_CUDA if the stream reports an error, else FP4Q_OK.
 * This is the only call that blocks the host.
 */
FP4Q_API int fp4q_device_status(fp4q_stream_t stream);

/*
 * fp4q_test_gemm_wait_timeout — failure-detection test of the bounded waits. The pages have no
 * counterpart: it exercises the library's own failure path without faulting the GPU.
 * Launches the CTA-pair MXFP8 GEMM kernel of fp4q_gemm_mxfp8 (fp32 output) on the given
 * operands with its producers issuing no copies, so no pipeline barrier ever completes: every
 * mbarrier wait of the kernel gives up after wait_limit_ns, raises the device error word and
 * ends its role; the kernel frees its tensor memory and returns with no copy in flight. d is
 * left unwritten. The next fp4q_device_status on the stream returns FP4Q_ERR_TIMEOUT (and
 * clears the word); later calls run normally.
 *   wait_limit_ns in [1e6, 2e9] (else FP4Q_ERR_ARG); the kernel takes a few limits in all.
 *   Shapes as fp4q_gemm_mxfp8 with M > 128 and K % 512 == 0 (the pair kernel's), 16-byte
 *   aligned pointers; a, a_scales, b, b_scales and d must be valid device buffers of those
 *   shapes (their tensor maps are built as for a real GEMM; nothing is read or written).
 */
FP4Q_API int fp4q_test_gemm_wait_timeout(const uint8_t* a, const uint8_t* a_scales,
                    const uint8_t* b, const uint8_t* b_scales, void* d,
                    int64_t M, int64_t N, int64_t K, int64_t wait_limit_ns, fp4q_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H */
