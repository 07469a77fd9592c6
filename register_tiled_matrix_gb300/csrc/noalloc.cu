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
// reads before reading it, so nothing needs clearing, but two calls in flight
// on the GPU at the same time (for example on two streams) race on it.
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_scratch_mutex;
float *g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// Set-up, once per device, with that device current: look up the device
// address of the scratch array (in host code the array's name is only a
// stand-in for it, not an address the GPU can use).
int scratch_for_current_device(float **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        float *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return GEMM_OK;
}

} // namespace

extern "C" int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                                float *C, void *stream)
{
    // The same host-side checks as gemm_f32, before any CUDA call.
    bool nothing = false;
    int st = rtm::check_f32_args(M, N, K, A, B, C, &nothing);
    if (st != GEMM_OK || nothing)
        return st;
    float *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != GEMM_OK)
        return st;
    // gemm_f32_ws over the built-in array: it splits K through the array when
    // the split fits in it, and otherwise runs gemm_f32's schedule (K split over
    // cluster CTAs, or none), which needs no scratch at all.
    return gemm_f32_ws(M, N, K, A, B, C, scratch, kScratchBytes, stream);
}
