// noalloc.cu — fp4q_quantize_2d_noalloc: the 16x16-tile NVFP4 weight quantizer for callers
// that cannot allocate device memory.
//
// fp4q_quantize_2d needs a small device workspace for the per-tensor amax values (one float
// per tensor of the batch). Some callers have no way to provide it: a plugin whose host
// framework owns every device allocation and hands out no workspace, or a latency-critical
// caller that must not call cudaMalloc because it can synchronize the whole device. This entry
// point keeps that workspace in a fixed array compiled into the library instead, so the caller
// passes only its inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's contents; the amax
// pass clears the part it uses before accumulating into it. Two calls whose work overlaps on
// the GPU (e.g. on two streams without ordering between them) race on the array.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include "../../include/fp4q.h"
#include "fp4q_internal.h"

namespace {

// One float per tensor of the batch: 1024 experts at most, 4 KiB per device, held by every
// GPU that loads the library until the process exits.
static __device__ __align__(256) float g_noalloc_amax[FP4Q_NOALLOC_MAX_BATCH];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_addr[kMaxDevices] = {nullptr};
void* g_scratch_ctx[kMaxDevices] = {nullptr};

// The current context of the calling thread (driver entry point, looked up once), or NULL.
void* current_context() {
    typedef int (*CtxGetCurrentFn)(void**);
    static CtxGetCurrentFn fn = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
        looked_up = true;
    }
    void* ctx = nullptr;
    if (fn && fn(&ctx) != 0) ctx = nullptr;
    return ctx;
}

// The device address of the array for the current device, looked up with that device current
// the first time it is used and again whenever the device's context has changed since (after a
// cudaDeviceReset the module is loaded anew and the array may sit elsewhere). In host code the
// array's name is only a host-side stand-in, so the kernels must be given this address.
int scratch_for_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP4Q_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP4Q_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    void* ctx = current_context();
    if (!g_scratch_addr[dev] || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess || !p) return FP4Q_ERR_CUDA;
        g_scratch_addr[dev] = static_cast<float*>(p);
        g_scratch_ctx[dev] = current_context();   // the lookup may have made the primary context current
    }
    *out = g_scratch_addr[dev];
    return FP4Q_OK;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fp4q_quantize_2d_noalloc(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                                        int64_t batch, int64_t batch_stride,
                                        uint8_t* codes, uint8_t* tile_scales, float* s_dec_out,
                                        fp4q_stream_t stream) {
    if (!w_bf16 || !codes || !tile_scales || !s_dec_out) return FP4Q_ERR_NULL;
    if (batch < 1 || batch > FP4Q_NOALLOC_MAX_BATCH) return FP4Q_ERR_SHAPE;   // beyond the fixed array
    if (rows < 16 || cols < 16 || rows % 16 != 0 || cols % 16 != 0 || ld < cols) return FP4Q_ERR_SHAPE;
    if (batch > 1 && batch_stride < rows * ld) return FP4Q_ERR_SHAPE;
    if (rows / 16 > 65535) return FP4Q_ERR_SHAPE;
    if (!al16(w_bf16) || ld % 8 != 0 || batch_stride % 8 != 0 || !al16(codes)) return FP4Q_ERR_ALIGN;
    if (int dv = fp4q::check_device()) return dv;
    float* amax = nullptr;
    if (int s = scratch_for_current_device(&amax)) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the amax pass zeroes amax[0, batch) on the stream, then accumulates into it
    if (fp4q::launch_amax(static_cast<const uint16_t*>(w_bf16), rows, cols, ld, batch, batch_stride, amax, st) !=
        cudaSuccess)
        return FP4Q_ERR_CUDA;
    return fp4q::launch_quantize_2d(static_cast<const uint16_t*>(w_bf16), rows, cols, ld, batch, batch_stride,
                                    amax, codes, tile_scales, s_dec_out, st) == cudaSuccess
               ? FP4Q_OK
               : FP4Q_ERR_CUDA;
}
