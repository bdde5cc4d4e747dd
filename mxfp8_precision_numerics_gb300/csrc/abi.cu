// abi.cu — the extern "C" entry points of libfp4q.so (declared and documented in
// include/fp4q.h): host-side argument validation, then the launches on the caller's stream.
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/fp4q.h"
#include "fp4q_internal.h"

namespace fp4q {

int num_sms() {
    static int cached_dev = -1, cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev != cached_dev) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        cached = n;
        cached_dev = dev;
    }
    return cached;
}

// The E2M1 conversion path: the hardware cvt.rn.satfinite.e2m1x2 (one instruction per two
// values). A device test checks it against the oracle's round-to-nearest-even rule on every
// tie of the grid, on saturation and on a dense sweep; the ALU rule stays as the reference.
bool use_hw_e2m1() { return true; }

// The kernels use tcgen05 / TMA instructions of compute capability 10.x.
int check_device() {
    static int cached_dev = -1, cached = FP4Q_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP4Q_ERR_CUDA;
    if (dev != cached_dev) {
        int major = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
            return FP4Q_ERR_CUDA;
        cached = (major == 10) ? FP4Q_OK : FP4Q_ERR_UNSUPPORTED;
        cached_dev = dev;
    }
    return cached;
}

}  // namespace fp4q

namespace {

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA; }

using fp4q::check_device;


}  // namespace

extern "C" {

const char* fp4q_status_str(int status) {
    switch (status) {
        case FP4Q_OK: return "FP4Q_OK";
        case FP4Q_ERR_NULL: return "FP4Q_ERR_NULL: a required pointer is NULL";
        case FP4Q_ERR_ALIGN: return "FP4Q_ERR_ALIGN: a pointer or leading dimension is misaligned";
        case FP4Q_ERR_SHAPE: return "FP4Q_ERR_SHAPE: a size is not allowed";
        case FP4Q_ERR_ARG: return "FP4Q_ERR_ARG: an enum or flag argument is out of range";
        case FP4Q_ERR_CUDA: return "FP4Q_ERR_CUDA: a CUDA call failed";
        case FP4Q_ERR_TIMEOUT: return "FP4Q_ERR_TIMEOUT: a bounded device-side wait gave up";
        case FP4Q_ERR_UNSUPPORTED: return "FP4Q_ERR_UNSUPPORTED: the device is not compute capability 10.x";
        default: return "FP4Q: unknown status";
    }
}

int fp4q_version(void) { return 100; }

int fp4q_quantize_1d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                     const float* amax_in, float* amax_ws,
                     uint8_t* codes, uint8_t* scales, float* s_dec_out, fp4q_stream_t stream) {
    if (!x_bf16 || !codes || !scales || !s_dec_out || (!amax_in && !amax_ws)) return FP4Q_ERR_NULL;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || ld < cols) return FP4Q_ERR_SHAPE;
    if (!al16(x_bf16) || ld % 8 != 0 || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const float* amax = amax_in;
    if (!amax) {
        cudaError_t e = fp4q::launch_amax(static_cast<const uint16_t*>(x_bf16), rows, cols, ld, 1, 0, amax_ws, st);
        if (e != cudaSuccess) return FP4Q_ERR_CUDA;
        amax = amax_ws;
    }
    return cuda_status(fp4q::launch_quantize_1d(static_cast<const uint16_t*>(x_bf16), rows, cols, ld, amax,
                                                codes, scales, s_dec_out, st));
}

int fp4q_quantize_1d_rows(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, int four_six,
                          uint8_t* codes, uint8_t* scales, float* s_dec_rows, fp4q_stream_t stream) {
    if (four_six != 0 && four_six != 1) return FP4Q_ERR_ARG;
    if (!x_bf16 || !codes || !scales || !s_dec_rows) return FP4Q_ERR_NULL;
    if (rows < 1 || cols < 16 || cols % 16 != 0 || ld < cols) return FP4Q_ERR_SHAPE;
    if (!al16(x_bf16) || ld % 8 != 0 || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    return cuda_status(fp4q::launch_quantize_1d_rows(static_cast<const uint16_t*>(x_bf16), rows, cols, ld,
                                                     four_six, codes, scales, s_dec_rows,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_quantize_2d(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                     int64_t batch, int64_t batch_stride,
                     const float* amax_in, float* amax_ws,
                     uint8_t* codes, uint8_t* tile_scales, float* s_dec_out,
                     fp4q_stream_t stream) {
    if (!w_bf16 || !codes || !tile_scales || !s_dec_out || (!amax_in && !amax_ws)) return FP4Q_ERR_NULL;
    if (rows < 16 || cols < 16 || rows % 16 != 0 || cols % 16 != 0 || ld < cols || batch < 1 || batch > 65535)
        return FP4Q_ERR_SHAPE;
    if (batch > 1 && batch_stride < rows * ld) return FP4Q_ERR_SHAPE;
    if (rows / 16 > 65535) return FP4Q_ERR_SHAPE;
    if (!al16(w_bf16) || ld % 8 != 0 || batch_stride % 8 != 0 || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const float* amax = amax_in;
    if (!amax) {
        cudaError_t e = fp4q::launch_amax(static_cast<const uint16_t*>(w_bf16), rows, cols, ld, batch,
                                          batch_stride, amax_ws, st);
        if (e != cudaSuccess) return FP4Q_ERR_CUDA;
        amax = amax_ws;
    }
    return cuda_status(fp4q::launch_quantize_2d(static_cast<const uint16_t*>(w_bf16), rows, cols, ld, batch,
                                                batch_stride, amax, codes, tile_scales, s_dec_out, st));
}

int fp4q_requant_t_mxfp8_sr(int in_kind, const void* in, const uint8_t* in_scales,
                            const float* in_s_dec, int64_t rows, int64_t cols,
                            int transpose, int rht, uint32_t rht_signs,
                            int rounding, uint64_t seed, uint32_t tensor_tag,
                            uint8_t* out_e4m3, uint8_t* out_e8m0, fp4q_stream_t stream) {
    if (in_kind < FP4Q_IN_BF16 || in_kind > FP4Q_IN_NVFP4_1D_ROWS) return FP4Q_ERR_ARG;
    if ((transpose != 0 && transpose != 1) || (rht != 0 && rht != 1)) return FP4Q_ERR_ARG;
    if (rounding != FP4Q_RNE && rounding != FP4Q_SR) return FP4Q_ERR_ARG;
    if (rht_signs > 0xFFFFu) return FP4Q_ERR_ARG;
    if (!in || !out_e4m3 || !out_e8m0) return FP4Q_ERR_NULL;
    if (in_kind != FP4Q_IN_BF16 && (!in_scales || !in_s_dec)) return FP4Q_ERR_NULL;
    if (rows < 32 || cols < 32 || rows % 32 != 0 || cols % 32 != 0) return FP4Q_ERR_SHAPE;
    if (transpose && (rows / 64 + 1 > 65535 || cols / 64 + 1 > 2147483647)) return FP4Q_ERR_SHAPE;
    if (!al16(in) || !al16(out_e4m3)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    fp4q::RequantArgs a;
    a.in_kind = in_kind;
    a.in = in;
    a.in_scales = in_scales;
    a.in_s_dec = in_s_dec;
    a.rows = rows;
    a.cols = cols;
    a.transpose = transpose;
    a.rht = rht;
    a.rht_signs = rht_signs;
    a.rounding = rounding;
    a.seed = seed;
    a.tag = tensor_tag;
    a.out_e4m3 = out_e4m3;
    a.out_e8m0 = out_e8m0;
    return cuda_status(fp4q::launch_requant(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_requant_bf16_dual(const void* in, int64_t rows, int64_t cols, int rht, uint32_t rht_signs,
                           int rounding, uint64_t seed, uint32_t tag_rows, uint32_t tag_t,
                           uint8_t* rows_e4m3, uint8_t* rows_e8m0, uint8_t* t_e4m3, uint8_t* t_e8m0,
                           fp4q_stream_t stream) {
    if (rht != 0 && rht != 1) return FP4Q_ERR_ARG;
    if (rounding != FP4Q_RNE && rounding != FP4Q_SR) return FP4Q_ERR_ARG;
    if (rht_signs > 0xFFFFu) return FP4Q_ERR_ARG;
    if (!in || !rows_e4m3 || !rows_e8m0 || !t_e4m3 || !t_e8m0) return FP4Q_ERR_NULL;
    if (rows < 32 || cols < 32 || rows % 32 != 0 || cols % 32 != 0) return FP4Q_ERR_SHAPE;
    if (rows / 64 + 1 > 65535 || cols / 64 + 1 > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(in) || !al16(rows_e4m3) || !al16(t_e4m3)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    fp4q::RequantArgs a;
    a.in_kind = FP4Q_IN_BF16;
    a.in = in;
    a.in_scales = nullptr;
    a.in_s_dec = nullptr;
    a.rows = rows;
    a.cols = cols;
    a.transpose = 1;
    a.rht = rht;
    a.rht_signs = rht_signs;
    a.rounding = rounding;
    a.seed = seed;
    a.tag = tag_t;
    a.out_e4m3 = t_e4m3;
    a.out_e8m0 = t_e8m0;
    a.out2_e4m3 = rows_e4m3;
    a.out2_e8m0 = rows_e8m0;
    a.tag2 = tag_rows;
    return cuda_status(fp4q::launch_requant(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_rht16(const void* in, int in_dtype, float* out, int64_t rows, int64_t cols,
               uint32_t signs, fp4q_stream_t stream) {
    if (in_dtype != FP4Q_F32 && in_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (signs > 0xFFFFu) return FP4Q_ERR_ARG;
    if (!in || !out) return FP4Q_ERR_NULL;
    if (rows < 1 || cols < 16 || cols % 16 != 0) return FP4Q_ERR_SHAPE;
    if (!al16(in) || !al16(out)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    return cuda_status(fp4q::launch_rht16(in, in_dtype == FP4Q_BF16, out, rows, cols, signs,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

static int validate_groups(int groups, const int64_t* offs, int64_t M) {
    if (groups < 1 || groups > 64) return FP4Q_ERR_ARG;
    if (groups == 1) return FP4Q_OK;
    if (!offs) return FP4Q_ERR_NULL;
    if (offs[0] != 0 || offs[groups] != M) return FP4Q_ERR_SHAPE;
    for (int g = 0; g < groups; ++g)
        if (offs[g + 1] < offs[g]) return FP4Q_ERR_SHAPE;
    return FP4Q_OK;
}

// a_rows: a_s_dec holds one outer scale per row of A (M floats) instead of one
static int gemm_nvfp4_impl(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec, int a_rows,
                           const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                           const float* b_s_dec, void* d, int d_dtype,
                           int64_t M, int64_t N, int64_t K,
                           int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream) {
    if (b_scale_kind != FP4Q_SCALE_1D && b_scale_kind != FP4Q_SCALE_2D) return FP4Q_ERR_ARG;
    if (d_dtype != FP4Q_F32 && d_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (!a || !a_scales || !a_s_dec || !b || !b_scales || !b_s_dec || !d) return FP4Q_ERR_NULL;
    if (int v = validate_groups(groups, group_row_offsets_host, M)) return v;
    if (M < 1 || N < 16 || N % 16 != 0 || K < 256 || K % 256 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N * groups > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al16(a_scales) || !al16(b_scales) || !al16(d)) return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 0;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = a_s_dec;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = b_scale_kind;
    g.b_s_dec = b_s_dec;
    g.d = d;
    g.d_bf16 = d_dtype == FP4Q_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = groups;
    g.group_offsets = group_row_offsets_host;
    g.a_sdec_rows = a_rows;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_gemm_nvfp4(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                    const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                    const float* b_s_dec, void* d, int d_dtype,
                    int64_t M, int64_t N, int64_t K,
                    int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream) {
    return gemm_nvfp4_impl(a, a_scales, a_s_dec, 0, b, b_scales, b_scale_kind, b_s_dec, d, d_dtype,
                           M, N, K, groups, group_row_offsets_host, stream);
}

int fp4q_gemm_nvfp4_rows(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec_rows,
                         const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                         const float* b_s_dec, void* d, int d_dtype,
                         int64_t M, int64_t N, int64_t K,
                         int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream) {
    return gemm_nvfp4_impl(a, a_scales, a_s_dec_rows, 1, b, b_scales, b_scale_kind, b_s_dec, d, d_dtype,
                           M, N, K, groups, group_row_offsets_host, stream);
}

int fp4q_gemm_nvfp4_combine(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                            const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                            const float* b_s_dec, uint32_t rht_signs, uint8_t* codes_out, uint8_t* e8m0_out,
                            int64_t M, int64_t N, int64_t K,
                            int groups, const int64_t* group_row_offsets_host, fp4q_stream_t stream) {
    if (b_scale_kind != FP4Q_SCALE_1D && b_scale_kind != FP4Q_SCALE_2D) return FP4Q_ERR_ARG;
    if (!a || !a_scales || !a_s_dec || !b || !b_scales || !b_s_dec || !codes_out || !e8m0_out) return FP4Q_ERR_NULL;
    if (int v = validate_groups(groups, group_row_offsets_host, M)) return v;
    if (M < 1 || N < 32 || N % 32 != 0 || K < 256 || K % 256 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N * groups > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al16(a_scales) || !al16(b_scales) || !al16(codes_out)) return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 0;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = a_s_dec;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = b_scale_kind;
    g.b_s_dec = b_s_dec;
    g.d = codes_out;
    g.d_bf16 = 0;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = groups;
    g.group_offsets = group_row_offsets_host;
    g.epi = 3;
    g.d2 = e8m0_out;
    g.rht32_signs = rht_signs;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_quantize_mxfp4(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, int rht, uint32_t rht_signs,
                        uint8_t* codes, uint8_t* e8m0, fp4q_stream_t stream) {
    if (rht != 0 && rht != 1) return FP4Q_ERR_ARG;
    if (!x_bf16 || !codes || !e8m0) return FP4Q_ERR_NULL;
    if (rows < 1 || cols < 32 || cols % 32 != 0 || ld < cols) return FP4Q_ERR_SHAPE;
    if (!al16(x_bf16) || ld % 8 != 0 || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    return cuda_status(fp4q::launch_quantize_mxfp4(static_cast<const uint16_t*>(x_bf16), rows, cols, ld, rht,
                                                   rht_signs, codes, e8m0, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_gemm_mxfp4(const uint8_t* a, const uint8_t* a_e8m0, const uint8_t* b, const uint8_t* b_e8m0,
                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K, fp4q_stream_t stream) {
    if (d_dtype != FP4Q_F32 && d_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (!a || !a_e8m0 || !b || !b_e8m0 || !d) return FP4Q_ERR_NULL;
    if (M < 1 || N < 16 || N % 16 != 0 || K < 2048 || K % 2048 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al16(a_e8m0) || !al16(b_e8m0) || !al16(d)) return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 2;
    g.a = a;
    g.a_scales = a_e8m0;
    g.a_s_dec = nullptr;
    g.b = b;
    g.b_scales = b_e8m0;
    g.b_scale_kind = 1;
    g.b_s_dec = nullptr;
    g.d = d;
    g.d_bf16 = d_dtype == FP4Q_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = 1;
    g.group_offsets = nullptr;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_combine_encode(const void* x, int x_dtype, int64_t rows, int64_t cols, uint32_t rht_signs,
                        uint8_t* codes, uint8_t* e8m0, fp4q_stream_t stream) {
    if (x_dtype != FP4Q_F32 && x_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (!x || !codes || !e8m0) return FP4Q_ERR_NULL;
    if (rows < 1 || cols < 32 || cols % 32 != 0) return FP4Q_ERR_SHAPE;
    if (!al16(x) || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    return cuda_status(fp4q::launch_combine_encode(x, x_dtype == FP4Q_BF16, rows, cols, rht_signs, codes, e8m0,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_combine_decode(const uint8_t* codes, const uint8_t* e8m0, int64_t tokens, int64_t k, int64_t cols,
                        uint32_t rht_signs, void* out, int out_dtype, fp4q_stream_t stream) {
    if (out_dtype != FP4Q_F32 && out_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (!codes || !e8m0 || !out) return FP4Q_ERR_NULL;
    if (tokens < 1 || k < 1 || cols < 32 || cols % 32 != 0) return FP4Q_ERR_SHAPE;
    if (!al16(codes) || !al16(out)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    return cuda_status(fp4q::launch_combine_decode(codes, e8m0, tokens, k, cols, rht_signs, out,
                                                   out_dtype == FP4Q_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_gemm_mxfp8(const uint8_t* a, const uint8_t* a_scales,
                    const uint8_t* b, const uint8_t* b_scales,
                    void* d, int d_dtype, int64_t M, int64_t N, int64_t K,
                    fp4q_stream_t stream) {
    if (d_dtype != FP4Q_F32 && d_dtype != FP4Q_BF16) return FP4Q_ERR_ARG;
    if (!a || !a_scales || !b || !b_scales || !d) return FP4Q_ERR_NULL;
    if (M < 1 || N < 16 || N % 16 != 0 || K < 128 || K % 128 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al4(a_scales) || !al4(b_scales) || !al16(d)) return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 1;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = nullptr;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = 1;
    g.b_s_dec = nullptr;
    g.d = d;
    g.d_bf16 = d_dtype == FP4Q_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = 1;
    g.group_offsets = nullptr;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_test_gemm_wait_timeout(const uint8_t* a, const uint8_t* a_scales,
                                const uint8_t* b, const uint8_t* b_scales, void* d,
                                int64_t M, int64_t N, int64_t K, int64_t wait_limit_ns,
                                fp4q_stream_t stream) {
    if (!a || !a_scales || !b || !b_scales || !d) return FP4Q_ERR_NULL;
    if (wait_limit_ns < 1000000 || wait_limit_ns > 2000000000) return FP4Q_ERR_ARG;
    // the CTA-pair kernel's shapes: more than one 128-row tile, whole scale units of 4 K-blocks
    if (M <= 128 || N < 16 || N % 16 != 0 || K < 512 || K % 512 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al16(a_scales) || !al16(b_scales) || !al16(d)) return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 1;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = nullptr;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = 1;
    g.b_s_dec = nullptr;
    g.d = d;
    g.d_bf16 = 0;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = 1;
    g.group_offsets = nullptr;
    g.wait_limit_ns = wait_limit_ns;
    g.no_copies = 1;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

// a_rows: per-row outer scales of A (act_amax may then be NULL)
static int gemm_nvfp4_gelu_impl(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec, int a_rows,
                                const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                                const float* b_s_dec, void* h_out, void* act_out, float* act_amax,
                                int64_t M, int64_t N, int64_t K, fp4q_stream_t stream) {
    if (b_scale_kind != FP4Q_SCALE_1D && b_scale_kind != FP4Q_SCALE_2D) return FP4Q_ERR_ARG;
    if (!a || !a_scales || !a_s_dec || !b || !b_scales || !b_s_dec || !h_out || !act_out ||
        (!act_amax && !a_rows))
        return FP4Q_ERR_NULL;
    if (M < 1 || N < 16 || N % 16 != 0 || K < 256 || K % 256 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N > 2147483647) return FP4Q_ERR_SHAPE;
    if (b_scale_kind == FP4Q_SCALE_2D && N % 16 != 0) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al16(a_scales) || !al16(b_scales) || !al16(h_out) || !al16(act_out))
        return FP4Q_ERR_ALIGN;
    if (act_amax && !al4(act_amax)) return FP4Q_ERR_ALIGN;
    if (int d = check_device()) return d;
    fp4q::GemmArgs g;
    g.kind = 0;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = a_s_dec;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = b_scale_kind;
    g.b_s_dec = b_s_dec;
    g.d = h_out;
    g.d_bf16 = 1;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = 1;
    g.group_offsets = nullptr;
    g.epi = 1;
    g.d2 = act_out;
    g.amax_out = act_amax;
    g.a_sdec_rows = a_rows;
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_gemm_nvfp4_gelu(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec,
                         const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                         const float* b_s_dec, void* h_out, void* act_out, float* act_amax,
                         int64_t M, int64_t N, int64_t K, fp4q_stream_t stream) {
    return gemm_nvfp4_gelu_impl(a, a_scales, a_s_dec, 0, b, b_scales, b_scale_kind, b_s_dec, h_out, act_out,
                                act_amax, M, N, K, stream);
}

int fp4q_gemm_nvfp4_gelu_rows(const uint8_t* a, const uint8_t* a_scales, const float* a_s_dec_rows,
                              const uint8_t* b, const uint8_t* b_scales, int b_scale_kind,
                              const float* b_s_dec, void* h_out, void* act_out, float* act_amax,
                              int64_t M, int64_t N, int64_t K, fp4q_stream_t stream) {
    return gemm_nvfp4_gelu_impl(a, a_scales, a_s_dec_rows, 1, b, b_scales, b_scale_kind, b_s_dec, h_out,
                                act_out, act_amax, M, N, K, stream);
}

int fp4q_gemm_mxfp8_dgelu(const uint8_t* a, const uint8_t* a_scales,
                          const uint8_t* b, const uint8_t* b_scales, const void* h, void* dh_out,
                          int64_t M, int64_t N, int64_t K, fp4q_stream_t stream) {
    if (!a || !a_scales || !b || !b_scales || !h || !dh_out) return FP4Q_ERR_NULL;
    if (M < 1 || N < 16 || N % 16 != 0 || K < 128 || K % 128 != 0) return FP4Q_ERR_SHAPE;
    if (M > 2147483647 || N > 2147483647) return FP4Q_ERR_SHAPE;
    if (!al16(a) || !al16(b) || !al4(a_scales) || !al4(b_scales) || !al16(h) || !al16(dh_out))
        return FP4Q_ERR_ALIGN;
    if (int dv = check_device()) return dv;
    fp4q::GemmArgs g;
    g.kind = 1;
    g.a = a;
    g.a_scales = a_scales;
    g.a_s_dec = nullptr;
    g.b = b;
    g.b_scales = b_scales;
    g.b_scale_kind = 1;
    g.b_s_dec = nullptr;
    g.d = dh_out;
    g.d_bf16 = 1;
    g.M = M;
    g.N = N;
    g.K = K;
    g.groups = 1;
    g.group_offsets = nullptr;
    g.epi = 2;
    g.aux = static_cast<const uint16_t*>(h);
    return cuda_status(fp4q::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4q_device_status(fp4q_stream_t stream) {
    int flag = 0;
    if (fp4q::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), &flag) != 0)
        return FP4Q_ERR_CUDA;
    return flag ? FP4Q_ERR_TIMEOUT : FP4Q_OK;
}

}  // extern "C"
