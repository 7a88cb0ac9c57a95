// pkv_probe.cu -- measured issue rates of tcgen05.mma (kind::f16, which the
// chunked-prefill kernel is built on, and kind::tf32), M = 128, for the
// roofline of that kernel.  A diagnostic: no counterpart on the pages.
//
// One CTA per SM; one thread issues `iters` MMAs back to back into one TMEM
// accumulator (zero operands: A from TMEM or shared memory, B from shared
// memory in the K-major 128-byte-swizzled layout), commits, and every thread
// waits (bounded) for the commit.  SM 0's CTA reports the clocks it took.
#include "../../include/pkv.h"
#include "pkv_internal.h"
#include "pkv_tcgen05.h"

#include <cuda_runtime.h>

#include <cstdio>

using namespace pkv;
using namespace pkv::tc;

namespace {

constexpr int kProbeThreads = 128;
// A (16 KiB) and B (up to 32 KiB) in the first 64 KiB; the launch asks for
// 120 KiB so that one CTA fits per SM (each holds all 512 TMEM columns)
constexpr size_t kProbeSmem = 120 * 1024;
constexpr uint32_t kProbeCols = 512;
constexpr uint32_t kColA = 256;                  // A in TMEM: columns 256 .. 319

template <int N, bool kTS, bool kF16>
__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_kernel(int iters, unsigned long long *cycles,
                                                                     int32_t *err) {
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t mbar;
    __shared__ uint32_t tslot;
    const int t = threadIdx.x, warp = t >> 5;
    for (int i = t; i < (64 * 1024) / 16; i += kProbeThreads)
        reinterpret_cast<float4 *>(sm)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t == 0) mbar_init(smem_u32(&mbar), 1);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tslot), kProbeCols);
        tmem_relinquish();
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = tslot;
    if constexpr (kTS) {
        // zero A in TMEM: each warp its 32 lanes, 64 columns
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        tmem_st32(tb + lane_base + kColA, z);
        tmem_st32(tb + lane_base + kColA + 32, z);
        tmem_st_wait();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    const unsigned long long c0 = clock64();
    if (t == 0) {
        const uint64_t ad = desc_sw128(smem_u32(sm)), bd = desc_sw128(smem_u32(sm + 16384));
        const uint32_t id = kF16 ? idesc_f16(128, N) : idesc_tf32(128, N);
#pragma unroll 1
        for (int i = 0; i < iters; i += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t acc = (i + j) > 0 ? 1u : 0u;
                if constexpr (kF16) {
                    if constexpr (kTS) mma_f16_ts(tb, tb + kColA + 8 * (j & 7), bd, id, acc);
                    else mma_f16(tb, ad, bd, id, acc);
                } else {
                    if constexpr (kTS) mma_tf32_ts(tb, tb + kColA + 8 * (j & 7), bd, id, acc);
                    else mma_tf32(tb, ad, bd, id, acc);
                }
            }
        }
        mma_commit(smem_u32(&mbar));
    }
    const bool ok = __syncthreads_and(mbar_wait(smem_u32(&mbar), 0));
    const unsigned long long c1 = clock64();
    if (t == 0) {
        if (!ok) atomicOr(err, static_cast<int32_t>(PKV_DEVERR_TIMEOUT));
        cycles[blockIdx.x] = c1 - c0;
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kProbeCols);
}

template <int N, bool kTS, bool kF16>
cudaError_t run_probe(int nsm, int iters, unsigned long long *dc, int32_t *de, float *ms) {
    static PerDeviceOnce configured;  // the attribute is per function and device
    cudaError_t e = configured.run([&]() -> cudaError_t {
        return cudaFuncSetAttribute(mma_rate_kernel<N, kTS, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kProbeSmem));
    });
    if (e != cudaSuccess) return e;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) {
        // warm-up, then the timed launch
        mma_rate_kernel<N, kTS, kF16><<<nsm, kProbeThreads, kProbeSmem>>>(64, dc, de);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventRecord(e0);
        if (e == cudaSuccess) {
            mma_rate_kernel<N, kTS, kF16><<<nsm, kProbeThreads, kProbeSmem>>>(iters, dc, de);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) e = cudaEventRecord(e1);
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return e;
}

// Both probes: kind::tf32 (K = 8 per MMA) or kind::f16 (K = 16).
template <bool kF16>
int probe_mma(int32_t n_cols, int32_t a_in_tmem, int32_t iters, double *clk_per_mma, double *tflops) {
    if (!clk_per_mma || !tflops) return report_error(PKV_ERR_ARG, "NULL output pointer");
    if (n_cols != 64 && n_cols != 128 && n_cols != 256)
        return report_error(PKV_ERR_ARG, "n_cols must be 64, 128 or 256");
    if (iters < 16 || iters > (1 << 20) || (iters % 16) != 0)
        return report_error(PKV_ERR_ARG, "iters must be a multiple of 16 in [16, 1048576]");
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return report_error(PKV_ERR_CUDA, cudaGetErrorString(e));
    unsigned long long *dc = nullptr;
    int32_t *de = nullptr;
    e = cudaMalloc(&dc, sizeof(unsigned long long) * nsm);
    if (e == cudaSuccess) e = cudaMalloc(&de, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(de, 0, sizeof(int32_t));
    float ms = 0.f;
    if (e == cudaSuccess) {
        const bool ts = a_in_tmem != 0;
        if (n_cols == 64)
            e = ts ? run_probe<64, true, kF16>(nsm, iters, dc, de, &ms) : run_probe<64, false, kF16>(nsm, iters, dc, de, &ms);
        else if (n_cols == 128)
            e = ts ? run_probe<128, true, kF16>(nsm, iters, dc, de, &ms) : run_probe<128, false, kF16>(nsm, iters, dc, de, &ms);
        else
            e = ts ? run_probe<256, true, kF16>(nsm, iters, dc, de, &ms) : run_probe<256, false, kF16>(nsm, iters, dc, de, &ms);
    }
    unsigned long long cyc = 0;
    int32_t he = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&cyc, dc, sizeof cyc, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&he, de, sizeof he, cudaMemcpyDeviceToHost);
    if (dc) cudaFree(dc);
    if (de) cudaFree(de);
    if (e != cudaSuccess) return report_error(PKV_ERR_CUDA, cudaGetErrorString(e));
    if (he) return report_error(PKV_ERR_DEVICE_TIMEOUT, "the probe's wait for its MMAs ran out");
    const double k = kF16 ? 16.0 : 8.0;
    *clk_per_mma = static_cast<double>(cyc) / iters;
    *tflops = 2.0 * 128.0 * n_cols * k * iters * nsm / (static_cast<double>(ms) * 1e-3) / 1e12;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_probe_tf32_mma(int32_t n_cols, int32_t a_in_tmem, int32_t iters, double *clk_per_mma,
                                  double *tflops) {
    return probe_mma<false>(n_cols, a_in_tmem, iters, clk_per_mma, tflops);
}

extern "C" int pkv_probe_f16_mma(int32_t n_cols, int32_t a_in_tmem, int32_t iters, double *clk_per_mma,
                                 double *tflops) {
    return probe_mma<true>(n_cols, a_in_tmem, iters, clk_per_mma, tflops);
}
