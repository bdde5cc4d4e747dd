// mma_ceiling.cu — the tensor-core ceiling of the library's GEMM instructions on this GPU: one
// thread per CTA (pair) issues the block-scaled tcgen05.mma forms the GEMMs use back to back, on
// operands already in shared memory and scales already in tensor memory (no loads, no epilogue),
// on every SM. Prints per form: kernel time, TFLOP/s, and the wall-clock window of its timing
// loop (to bin nvidia-smi clock samples by form). A measurement tool, not part of the library:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o mma_ceiling mma_ceiling.cu
//   ./mma_ceiling
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <chrono>
#include <vector>
#include <algorithm>

__device__ unsigned int g_err;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t globaltimer() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ uint32_t cluster_rank() { uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{.reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// bounded spin on the non-blocking test
__device__ __forceinline__ bool mbar_wait_test(uint64_t* bar, uint32_t parity, uint64_t limit) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer() - t0 > limit) { atomicOr(&g_err, 1u); return false; }
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer() - t0 > limit) { atomicOr(&g_err, 1u); return false; }
    }
}
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// kind 0 NVFP4 (mxf4nvf4 4X, UE4M3), 1 MXFP8 (mxf8f6f4 1X, UE8M0), 2 MXFP4 (mxf4nvf4 2X, UE8M0)
template <int kKind, bool kPair>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                    uint32_t acc) {
    if (kPair) {
        if (kKind == 0)
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
        else if (kKind == 1)
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
        else
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    } else {
        if (kKind == 0)
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
        else if (kKind == 1)
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
        else
            asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
                         "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;}"
                         ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
    }
}

constexpr uint32_t kSmem = 200 * 1024;   // one CTA per SM

// kMode: 0 one commit at the end; 1 a commit after every K-block (4 MMAs); 2 two commits per
// K-block; 3 / 4 a commit per K-block and, before issuing K-block g, a wait for the completion of
// K-block g - 4 / g - 2 (the dependency a pipelined GEMM's stage reuse puts on the issuing thread);
// 5 the same wait on K-block g - 8 (long complete); 6 the wait on g - 4 by the non-blocking test;
// 7 two waits on long-complete K-blocks (g - 8, g - 7); 8 the wait on g - 4 between the K-block's
// second and third MMA; 9 two waits (g - 4, g - 3) there; 10 one wait after the second MMA and one
// after the third
template <int kKind, bool kPair, int kMode = 0>
__global__ void __launch_bounds__(128, 1) ceiling_kernel(int kblocks) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint64_t* done = reinterpret_cast<uint64_t*>(smem + 65536);
    uint64_t* cb = done + 1;                       // per-K-block commit barriers (kMode > 0)
    uint32_t* slot = reinterpret_cast<uint32_t*>(cb + 8);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = kPair ? cluster_rank() : 0;
    // operands: A 128 x 128 B at 0, B (pair: this CTA's 128 of 256 rows; single: 256 rows) at 16 KB
    for (int i = threadIdx.x; i < 65536 / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        for (int i = 0; i < 8; ++i) mbar_init(&cb[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        if (kPair) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(512));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(512));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (kPair) cluster_sync();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *slot;
    // scale columns 256 .. 303: UE4M3 1.0 (0x38) or UE8M0 1.0 (0x7F) in every byte
    const uint32_t sv = kKind == 0 ? 0x38383838u : 0x7F7F7F7Fu;
    for (int c = 0; c < 48; ++c) tmem_st32(tmem + ((uint32_t)(32 * warp) << 16) + 256 + c, sv);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (kPair) cluster_sync();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    constexpr uint32_t M = kPair ? 256 : 128;
    const uint32_t idesc = kKind == 1 ? ((0u << 7) | (0u << 10) | ((256u >> 3) << 17) | (1u << 23) | ((M >> 4) << 24))
                         : kKind == 0 ? ((1u << 7) | (1u << 10) | ((256u >> 3) << 17) | (0u << 23) | ((M >> 4) << 24))
                                      : ((1u << 7) | (1u << 10) | ((256u >> 3) << 17) | (1u << 23) | ((M >> 4) << 24));
    if (rank == 0 && threadIdx.x == 0) {
        const uint32_t sa = smem_u32(smem), sb = sa + 16384;
        const uint32_t sf = tmem + 256;
        constexpr int kDepth = kMode == 3 ? 4 : 2;
        for (int kb = 0; kb < kblocks; ++kb) {
            if ((kMode == 3 || kMode == 4) && kb >= kDepth) {
                const int g = kb - kDepth;
                if (!mbar_wait(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
            }
            if (kMode == 5 && kb >= 8) {
                const int g = kb - 8;
                if (!mbar_wait(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
            }
            if (kMode == 6 && kb >= 4) {
                const int g = kb - 4;
                if (!mbar_wait_test(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
            }
            if (kMode == 7 && kb >= 8) {
                const int g = kb - 8;
                if (!mbar_wait(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
                if (!mbar_wait(&cb[(g + 1) % 8], (uint32_t)((g + 1) / 8) & 1u, 10000000000ull)) break;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if ((kMode == 8 || kMode == 9 || kMode == 10) && j == 2 && kb >= 4) {
                    const int g = kb - 4;
                    if (!mbar_wait(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
                    if (kMode == 9 && !mbar_wait(&cb[(g + 1) % 8], (uint32_t)((g + 1) / 8) & 1u, 10000000000ull)) break;
                }
                if (kMode == 10 && j == 3 && kb >= 4) {
                    const int g = kb - 3;
                    if (!mbar_wait(&cb[g % 8], (uint32_t)(g / 8) & 1u, 10000000000ull)) break;
                }
                if (kKind == 0)
                    mma<0, kPair>(tmem, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j), idesc, sf + 4 * j,
                                  sf + 16 + 8 * j, (kb | j) ? 1u : 0u);
                else if (kKind == 2) {
                    const uint32_t id = 2u * (uint32_t)(j & 1);
                    mma<2, kPair>(tmem, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j), idesc | (id << 29) | (id << 4),
                                  sf + 4 * (j >> 1), sf + 8 + 8 * (j >> 1), (kb | j) ? 1u : 0u);
                } else
                    mma<1, kPair>(tmem, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j),
                                  idesc | ((uint32_t)j << 29) | ((uint32_t)j << 4), sf, sf + 4, (kb | j) ? 1u : 0u);
            }
            for (int c = 0; c < (kMode == 2 ? 2 : kMode > 0 ? 1 : 0); ++c) {   // one or two commits
                uint64_t* bar = c ? &cb[(kb % 8) ^ 4] : &cb[kb % 8];
                if (kPair)
                    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                                 ::"r"(smem_u32(bar)), "h"((unsigned short)3) : "memory");
                else
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 ::"r"(smem_u32(bar)) : "memory");
            }
        }
        if (kPair)
            asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                         ::"r"(smem_u32(done)), "h"((unsigned short)3) : "memory");
        else
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(smem_u32(done)) : "memory");
    }
    mbar_wait(done, 0, 10000000000ull);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    __syncthreads();
    if (kPair) cluster_sync();
    if (warp == 0) {
        if (kPair) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
        else asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

template <int kKind, bool kPair, int kMode = 0>
void run(const char* name, int sms, double seconds) {
    auto kern = ceiling_kernel<kKind, kPair, kMode>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    int ctas = kPair ? (sms / 2) * 2 : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    if (kPair) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(ctas);
        q.blockDim = dim3(128);
        q.dynamicSmemBytes = kSmem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        q.attrs = at;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess && n > 0 && 2 * n < ctas) ctas = 2 * n;
        cfg.gridDim = dim3(ctas);
    }
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int kblocks = 8192;
    // warm-up
    cudaLaunchKernelEx(&cfg, kern, kblocks);
    if (cudaDeviceSynchronize() != cudaSuccess) { printf("%s: error %s\n", name, cudaGetErrorString(cudaGetLastError())); return; }
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    // one batch ~ 50 ms, repeated for `seconds`
    std::vector<double> ms;
    auto w0 = std::chrono::system_clock::now();
    double total = 0;
    int batches = 0;
    while (total < seconds * 1e3) {
        cudaEventRecord(e0);
        for (int i = 0; i < 10; ++i) cudaLaunchKernelEx(&cfg, kern, kblocks);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        float t = 0;
        cudaEventElapsedTime(&t, e0, e1);
        ms.push_back(t / 10);
        total += t;
        ++batches;
    }
    auto w1 = std::chrono::system_clock::now();
    std::vector<double> s = ms;
    std::sort(s.begin(), s.end());
    const double med = s[s.size() / 2], best = s.front();
    const double kmma = kKind == 1 ? 32 : 64;
    const double mrow = kPair ? 256 : 128;
    const double units = kPair ? ctas / 2 : ctas;
    const double flop = units * kblocks * 4.0 * 2.0 * mrow * 256.0 * kmma;
    unsigned int err = 0;
    cudaMemcpyFromSymbol(&err, g_err, sizeof(err));
    printf("%-28s ctas %d kernel_ms med %.4f best %.4f  TFLOP/s med %.1f best %.1f  err %u  wall %.3f %.3f\n", name, ctas,
           med, best, flop / (med * 1e-3) / 1e12, flop / (best * 1e-3) / 1e12, err,
           std::chrono::duration<double>(w0.time_since_epoch()).count(),
           std::chrono::duration<double>(w1.time_since_epoch()).count());
    fflush(stdout);
}

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    printf("SMs %d\n", sms);
    run<1, true>("mxfp8 pair 256x256x32", sms, 1.5);
    run<0, true>("nvfp4 pair 256x256x64", sms, 1.5);
    run<2, true>("mxfp4 pair 256x256x64", sms, 1.5);
    run<1, false>("mxfp8 single 128x256x32", sms, 1.5);
    run<0, false>("nvfp4 single 128x256x64", sms, 1.5);
    run<2, false>("mxfp4 single 128x256x64", sms, 1.5);
    run<1, true>("mxfp8 pair 256x256x32 (again)", sms, 1.5);
    run<0, true>("nvfp4 pair 256x256x64 (again)", sms, 1.5);
    run<1, true, 1>("mxfp8 pair, commit / K-block", sms, 1.0);
    run<0, true, 1>("nvfp4 pair, commit / K-block", sms, 1.0);
    run<1, true, 2>("mxfp8 pair, 2 commits / K-block", sms, 1.0);
    run<0, true, 2>("nvfp4 pair, 2 commits / K-block", sms, 1.0);
    run<1, true, 3>("mxfp8 pair, wait K-block g-4", sms, 1.0);
    run<0, true, 3>("nvfp4 pair, wait K-block g-4", sms, 1.0);
    run<1, true, 4>("mxfp8 pair, wait K-block g-2", sms, 1.0);
    run<0, true, 4>("nvfp4 pair, wait K-block g-2", sms, 1.0);
    run<0, true, 5>("nvfp4 pair, wait K-block g-8", sms, 1.0);
    run<0, true, 6>("nvfp4 pair, test-wait K-block g-4", sms, 1.0);
    run<0, true, 7>("nvfp4 pair, 2 waits g-8, g-7", sms, 1.0);
    run<0, true, 8>("nvfp4 pair, wait g-4 after MMA 2", sms, 1.0);
    run<0, true, 9>("nvfp4 pair, 2 waits after MMA 2", sms, 1.0);
    run<0, true, 10>("nvfp4 pair, waits after MMA 2, 3", sms, 1.0);
    run<1, true, 8>("mxfp8 pair, wait g-4 after MMA 2", sms, 1.0);
    run<1, true, 10>("mxfp8 pair, waits after MMA 2, 3", sms, 1.0);
    return 0;
}
