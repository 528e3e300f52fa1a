// peak.cu -- measured issue rates of the instruction routes an exact int8
// product can take on this GPU, and the device's copy bandwidth: the
// denominators of the roofline fractions the library's benchmark reports.
//
// sm_103a has no integer kind of tcgen05.mma (ptxas rejects kind::i8 for it),
// so the convolution kernel forms int8 products exactly on the f16 path of
// tcgen05.mma.  The integer routes that remain are the warp-level
// mma.sync ... s8 instruction and the CUDA cores' 4-way dot product (dp4a).
// Each kernel here runs one of them back to back from registers or shared
// memory, long enough (about a millisecond) for CUDA events around the
// launch to time it, on every SM:
//   * tcgen05 kind::f16: one CTA per SM (its shared memory forbids a second);
//     one thread issues M=128 N=256 K=16 MMAs from shared-memory operands
//     into two tensor-memory accumulators in turn, then waits for their
//     completion on an mbarrier (bounded in time);
//   * mma.sync m16n8k32 s8 -> s32 and m16n8k16 f16 -> f32: 8 warps per
//     block, 4 blocks per SM, 8 independent accumulators per warp;
//   * dp4a: the same grid, 8 independent int32 accumulators per thread;
//   * copy: 16-byte loads and stores over two halves of a caller buffer.
// Operand values are small integers (the rates do not depend on them).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace i8c {
namespace {

constexpr int kTcThreads = 128;
constexpr int kTcM = 128, kTcN = 256, kTcK = 16;
constexpr int kTcABytes = kTcM * 128, kTcBBytes = kTcN * 128;  // one 128-byte swizzled row per M / N
constexpr int kTcSmem = 120 * 1024;  // above half an SM's shared memory: one CTA per SM
constexpr int kTcCols = 512;         // two accumulators of 256 columns
constexpr uint64_t kTcWaitNs = 2000000000ull;

// Clock records of CTA 0: cycles and nanoseconds between the first and the
// last MMA's completion.
struct TcClock {
    unsigned long long cycles, ns;
};

__global__ void __launch_bounds__(kTcThreads, 1) peak_tcgen05_f16_kernel(int iters, TcClock *clk, int *status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t done_bar;
    __shared__ uint32_t tmem_base_sh;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    // small integer f16 operands: (i % 7) - 3
    for (int i = threadIdx.x; i < (kTcABytes + kTcBBytes) / 2; i += blockDim.x)
        reinterpret_cast<__half *>(base_ptr)[i] = __int2half_rn((i % 7) - 3);
    ptx::fence_proxy_async_smem();
    const uint32_t bar = ptx::smem_addr(&done_bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(ptx::smem_addr(&tmem_base_sh), kTcCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    if (threadIdx.x == 0) {
        const uint64_t adesc = ptx::smem_desc_sw128(base);
        const uint64_t bdesc = ptx::smem_desc_sw128(base + kTcABytes);
        constexpr uint32_t idesc = ptx::idesc_f16_f32(kTcM, kTcN);
        const unsigned long long c0 = clock64();
        const uint64_t t0 = ptx::global_timer_ns();
        for (int i = 0; i < iters; ++i) {
            // K steps of 16 f16 (32 bytes) along the 128-byte rows, two accumulators in turn
            const uint64_t k = (uint64_t)(2 * (i & 3));
            ptx::mma_f16_ss(tmem + (uint32_t)((i & 1) * kTcN), adesc + k, bdesc + k, idesc, i > 1 ? 1u : 0u);
        }
        ptx::mma_commit(bar);
        bool ok = true;
        while (!ptx::mbar_try_wait(bar, 0)) {
            if (ptx::global_timer_ns() - t0 > kTcWaitNs) {
                ok = false;
                atomicExch(status, (int)CONV_ERR_DEVICE_TIMEOUT);
                break;
            }
        }
        if (!ok) {
            // let the issued MMAs finish before tensor memory is released
            const uint64_t t1 = ptx::global_timer_ns();
            while (!ptx::mbar_try_wait(bar, 0) && ptx::global_timer_ns() - t1 < kTcWaitNs) {
            }
        }
        if (blockIdx.x == 0 && clk) {
            clk->cycles = clock64() - c0;
            clk->ns = ptx::global_timer_ns() - t0;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (threadIdx.x < 32) ptx::tmem_dealloc(tmem, kTcCols);
}

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

constexpr int kChains = 8;  // independent accumulators per warp / thread

__global__ void __launch_bounds__(256) peak_mma_s8_kernel(int iters, int *sink) {
    uint32_t a[4], b[2];
    for (int i = 0; i < 4; ++i) a[i] = 0x01020301u * (threadIdx.x + i);
    for (int i = 0; i < 2; ++i) b[i] = 0x03010201u * (threadIdx.x + 3 * i);
    int32_t d[kChains][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) mma_s8(d[j], a, b);
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += d[j][0] + d[j][1] + d[j][2] + d[j][3];
    if (s == 0x7654321) sink[0] = s;  // keeps the results live
}

__global__ void __launch_bounds__(256) peak_mma_f16_kernel(int iters, int *sink) {
    uint32_t a[4], b[2];
    for (int i = 0; i < 4; ++i) a[i] = 0x3c003c00u ^ ((threadIdx.x + i) & 0x3ff);
    for (int i = 0; i < 2; ++i) b[i] = 0x3c003c00u ^ ((threadIdx.x + 5 * i) & 0x3ff);
    float d[kChains][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) mma_f16(d[j], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += d[j][0] + d[j][1] + d[j][2] + d[j][3];
    if (s == 1.2345f) sink[0] = 1;
}

__global__ void __launch_bounds__(256) peak_dp4a_kernel(int iters, int *sink) {
    const int a = (int)(0x01020304u * (threadIdx.x + 1)), b = (int)(0x04030201u ^ threadIdx.x);
    int d[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) d[j] = j;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kChains; ++j)
            asm volatile("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(d[j]) : "r"(a + j), "r"(b));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += d[j];
    if (s == 0x7654321) sink[0] = s;
}

__global__ void __launch_bounds__(256) peak_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                        int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// Best (shortest) of `reps` event-timed launches of `launch`, in ms.
template <class F>
conv_status best_ms(cudaStream_t st, int reps, F launch, float *out) {
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return CONV_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return CONV_ERR_CUDA;
    }
    conv_status rc = CONV_OK;
    float best = 0.f;
    for (int r = 0; r < reps && rc == CONV_OK; ++r) {
        cudaEventRecord(e0, st);
        launch();
        cudaEventRecord(e1, st);
        float ms = 0.f;
        if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
            rc = CONV_ERR_CUDA;
        else if (r == 0 || ms < best)
            best = ms;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *out = best;
    return rc;
}

}  // namespace
}  // namespace i8c

using namespace i8c;

extern "C" conv_status conv_measure_peak_rates(void *scratch, size_t scratch_bytes, conv_peak_rates *out,
                                               void *stream) {
    if (!out || !scratch) return CONV_ERR_NULL_PTR;
    if (scratch_bytes < ((size_t)1 << 20) || ((uintptr_t)scratch % 256) != 0) return CONV_ERR_WORKSPACE;
    conv_status st = check_device();
    if (st) return st;
    int *status = device_status_word();
    if (!status) return CONV_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const int sms = device_sm_count();
    uint8_t *buf = static_cast<uint8_t *>(scratch);
    TcClock *clk = reinterpret_cast<TcClock *>(buf);
    int *sink = reinterpret_cast<int *>(buf + 256);
    *out = conv_peak_rates{};

    // tcgen05 kind::f16, M=128 N=256 K=16 per instruction
    if (cudaFuncSetAttribute(peak_tcgen05_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) !=
        cudaSuccess)
        return CONV_ERR_CUDA;
    const int tc_iters = 16384;
    float ms = 0.f;
    st = best_ms(s, 3, [&] { peak_tcgen05_f16_kernel<<<sms, kTcThreads, kTcSmem, s>>>(tc_iters, clk, status); },
                 &ms);
    if (st) return st;
    out->tcgen05_f16_tflops = 2.0 * kTcM * kTcN * kTcK * (double)tc_iters * sms / (ms * 1e-3) / 1e12;
    TcClock c{};
    if (cudaMemcpy(&c, clk, sizeof(c), cudaMemcpyDeviceToHost) != cudaSuccess) return CONV_ERR_CUDA;
    out->sm_mhz = c.ns ? (double)c.cycles / (double)c.ns * 1e3 : 0.0;

    // warp-level MMAs and dp4a: 4 blocks of 8 warps per SM
    const int blocks = sms * 4, threads = 256, iters = 4096;
    const double warps = (double)blocks * (threads / 32);
    st = best_ms(s, 3, [&] { peak_mma_s8_kernel<<<blocks, threads, 0, s>>>(iters, sink); }, &ms);
    if (st) return st;
    out->mma_sync_s8_tops = 2.0 * 16 * 8 * 32 * (double)iters * kChains * warps / (ms * 1e-3) / 1e12;
    st = best_ms(s, 3, [&] { peak_mma_f16_kernel<<<blocks, threads, 0, s>>>(iters, sink); }, &ms);
    if (st) return st;
    out->mma_sync_f16_tflops = 2.0 * 16 * 8 * 16 * (double)iters * kChains * warps / (ms * 1e-3) / 1e12;
    st = best_ms(s, 3, [&] { peak_dp4a_kernel<<<blocks, threads, 0, s>>>(iters * 4, sink); }, &ms);
    if (st) return st;
    out->dp4a_tops = 8.0 * (double)iters * 4 * kChains * (double)blocks * threads / (ms * 1e-3) / 1e12;

    // copy over the rest of the buffer (when it is well above the L2 size)
    const size_t avail = scratch_bytes - 4096;
    if (avail >= ((size_t)512 << 20)) {
        const int64_t n = (int64_t)(avail / 2 / 16);
        const uint4 *src = reinterpret_cast<const uint4 *>(buf + 4096);
        uint4 *dst = reinterpret_cast<uint4 *>(buf + 4096 + (size_t)n * 16);
        st = best_ms(s, 5, [&] { peak_copy_kernel<<<sms * 8, 256, 0, s>>>(src, dst, n); }, &ms);
        if (st) return st;
        out->hbm_copy_gbs = 2.0 * 16.0 * (double)n / (ms * 1e-3) / 1e9;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return CONV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CONV_ERR_CUDA;
    return v ? (conv_status)v : CONV_OK;
}
