// gemm_f32_noalloc: the split-K fp32 product with its scratch memory built
// into the library, for callers that cannot allocate device memory.
//
// Who cannot allocate: code that runs inside a host application which owns
// all device memory through its own pool and forbids other allocations (a
// plugin, an embedded runtime), and code that must not be able to fail for
// lack of memory once it is loaded, because it has no way to report or
// recover from an out-of-memory error at call time. For them the split-K
// workspace that gemm_f32_ws takes from the caller lives here instead, in a
// fixed-size array reserved on every GPU that loads this library, until the
// process exits.
//
// The register-tiling pages have no counterpart of this entry point; it is a
// deployment convenience around the split-K schedule of the SIMT product.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "gemm.h"
#include "kernels.h"

constexpr int64_t kScratchBytes = 24ll << 20;  // 24 MiB per device

// The scratch: every partial product slab of a call lives here. Its contents
// persist from one call to the next; a call writes every element it later
// reads, so nothing needs clearing, but two calls in flight on the GPU at the
// same time (for example on two streams) race on it.
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;

struct ScratchInfo {
    bool ready = false;
    float *ptr = nullptr;  // device address of g_noalloc_scratch on this device
    int sms = 0;
    int cc = 0;
};

std::mutex g_scratch_mutex;
ScratchInfo g_scratch[kMaxDevices];

// Set-up, once per device, with that device current: look up the device
// address of the scratch array (in host code the array's name is only a
// stand-in for it) and the SM count the split plan depends on.
int scratch_for_current_device(ScratchInfo *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchInfo &s = g_scratch[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        float *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        s.ptr = ptr;
        s.sms = sms;
        s.cc = major * 10 + minor;
        s.ready = true;
    }
    *out = s;
    return s.cc == 103 ? GEMM_OK : GEMM_ERR_DEVICE;
}

bool ranges_overlap(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes)
{
    if (!a || !b || a_bytes <= 0 || b_bytes <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)b_bytes && b0 < a0 + (uintptr_t)a_bytes;
}

} // namespace

extern "C" int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                                float *C, void *stream)
{
    constexpr int64_t kMaxDim = 0x7fffffff;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (!C || (K > 0 && (!A || !B)))
        return GEMM_ERR_INVALID_ARG;
    if (M * N > (int64_t)1 << 52 || M * K > (int64_t)1 << 52 || K * N > (int64_t)1 << 52)
        return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (ranges_overlap(C, M * N * 4, A, M * K * 4) ||
                  ranges_overlap(C, M * N * 4, B, K * N * 4)))
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 3) != 0)))
        return GEMM_ERR_ALIGNMENT;

    ScratchInfo sc;
    int st = scratch_for_current_device(&sc);
    if (st != GEMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0) {
        e = rtm::launch_zero_fill(C, M * N, s);
    } else if (M <= rtm::kShortMaxM) {
        // Short, wide products split K over CTA clusters and need no scratch.
        e = rtm::launch_sgemm_short((int)M, (int)N, (int)K, A, B, C,
                                    rtm::sgemm_short_splits((int)M, (int)N, (int)K, sc.sms), s);
    } else {
        const rtm::F32Schedule f = rtm::sgemm_ws_schedule((int)M, (int)N, (int)K, sc.sms);
        const rtm::SplitK &plan = f.workspace;
        if (plan.splits <= 1) {
            e = rtm::launch_sgemm_f32_tiles((int)M, (int)N, (int)K, A, B, C, f.cluster, sc.sms, s);
        } else {
            if ((int64_t)plan.splits * M * N * (int64_t)sizeof(float) > kScratchBytes)
                return GEMM_ERR_INVALID_ARG;  // needs more than the fixed 24 MiB of scratch
            e = rtm::launch_sgemm_f32_splitk((int)M, (int)N, (int)K, A, B, C, plan, sc.ptr, s);
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}
