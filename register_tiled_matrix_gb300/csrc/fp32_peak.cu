// Throughput of this GPU's FP32 FMA pipes, measured: the denominator of the
// SIMT product's roofline.
//
// Every thread runs kChains independent FMA chains x <- x * a + b on values
// held in registers, so nothing but the FMA pipe is exercised: no memory
// traffic, no shared memory, and enough independent instructions in flight
// (kChains per warp, 8 warps per SM partition) to cover the FMA latency.
// The kernel also records, over its whole run, the SM clock cycles and the
// nanoseconds of the global timer elapsed in each CTA; the largest of each
// gives the clock the SMs actually ran at during the measurement.
//
// The register-tiling pages name the FP32 cores per SM as the resource the
// register tile feeds ("GPU架构基础", the SM and CUDA-core section); this
// kernel measures how fast those cores retire FMAs on GB300.
#include <cstdint>

#include <cuda_runtime.h>

#include "gemm.h"
#include "ptx.cuh"

namespace {

constexpr int kPeakThreads = 256;
constexpr int kPeakBlocksPerSm = 4;  // 1024 threads per SM: 8 warps per partition
constexpr int kChains = 16;          // independent accumulators per thread
constexpr int kUnroll = 32;          // chain steps per loop iteration (loop overhead < 1 %)

__device__ __forceinline__ long long clock_cycles()
{
    long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

// PACKED: the same chains as pairs through the packed FP32 FMA (two FMAs per
// instruction, fma.rn.f32x2).
template <bool PACKED>
__global__ void __launch_bounds__(kPeakThreads)
    ffma_peak_kernel(long long iters, float a, float b, unsigned long long *clock_out, float *sink)
{
    const uint64_t t0 = rtm::globaltimer_ns();
    const long long c0 = clock_cycles();
    float x[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        x[i] = (float)(threadIdx.x * kChains + i) * 1e-6f;
    if constexpr (PACKED) {
        float2 y[kChains / 2];
#pragma unroll
        for (int i = 0; i < kChains / 2; ++i)
            y[i] = make_float2(x[2 * i], x[2 * i + 1]);
        const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int i = 0; i < kChains / 2; ++i)
                    y[i] = __ffma2_rn(y[i], a2, b2);
        }
#pragma unroll
        for (int i = 0; i < kChains / 2; ++i) {
            x[2 * i] = y[i].x;
            x[2 * i + 1] = y[i].y;
        }
    } else {
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int i = 0; i < kChains; ++i)
                    x[i] = fmaf(x[i], a, b);
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        s += x[i];
    // The chains converge to b / (1 - a), a finite value; the store keeps
    // them live and is never taken for the arguments the host passes.
    if (s == -1.0f)
        sink[0] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long cycles = clock_cycles() - c0;
        const uint64_t ns = rtm::globaltimer_ns() - t0;
        atomicMax(clock_out, (unsigned long long)cycles);
        atomicMax(clock_out + 1, (unsigned long long)ns);
    }
}

} // namespace

extern "C" int gemm_fp32_pipe_peak(int64_t iters, int packed, unsigned long long *clock_out,
                                   double *flops, void *stream)
{
    if (iters < 1 || iters > ((int64_t)1 << 40) || !clock_out || !flops)
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(clock_out) & 7) != 0)
        return GEMM_ERR_ALIGNMENT;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (major * 10 + minor != 103)
        return GEMM_ERR_DEVICE;
    const int blocks = sms * kPeakBlocksPerSm;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a = 1 - 2^-20, b = 2^-20: every chain stays near 1 (no overflow, no
    // subnormals), so the FMA pipe runs at its normal-operand rate.
    const float a = 1.0f - 1.0f / 1048576.0f, b = 1.0f / 1048576.0f;
    // `sink` is only a store target that is never written (see the kernel).
    float *sink = reinterpret_cast<float *>(clock_out);
    if (packed)
        ffma_peak_kernel<true><<<blocks, kPeakThreads, 0, s>>>(iters, a, b, clock_out, sink);
    else
        ffma_peak_kernel<false><<<blocks, kPeakThreads, 0, s>>>(iters, a, b, clock_out, sink);
    if (cudaGetLastError() != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    *flops = 2.0 * (double)blocks * kPeakThreads * kChains * kUnroll * (double)iters;
    return GEMM_OK;
}
