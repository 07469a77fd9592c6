// C ABI of libgemm_gb300.so (declared in include/gemm.h).
//
// Host-side argument checks run before any CUDA call, so invalid arguments
// are reported without touching a device. The only library state is a
// per-device cache (compute capability, SM count) and one device error word
// per device, written by kernels whose bounded waits give up.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm.h"
#include "kernels.h"
#include "ptx.cuh"

namespace {

// Device error word: 0, or the status of the first bounded wait that gave up.
__device__ int g_device_error = 0;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;  // 4 s per wait

struct DeviceInfo {
    bool ready = false;
    int cc = 0;
    int sms = 0;
    int *err = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
void *g_encode_tiled = nullptr;
bool g_encode_tried = false;

// Both zero fills let a dependent kernel launched with programmatic stream
// serialization start at once (the CTA-pair kernel waits for the zeros only
// before its reduce-adds).
__global__ void zero_fill_kernel(float *C, int64_t count)
{
    rtm::grid_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
        C[i] = 0.0f;
}

__global__ void zero_fill4_kernel(float4 *C, int64_t count4)
{
    rtm::grid_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count4; i += stride)
        C[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Current device's cached info; GEMM_OK or an error status.
int current_device(DeviceInfo *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        void *err = nullptr;
        if (cudaGetSymbolAddress(&err, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        d.cc = major * 10 + minor;
        d.sms = sms;
        d.err = static_cast<int *>(err);
        d.ready = true;
    }
    *out = d;
    return d.cc == 103 ? GEMM_OK : GEMM_ERR_DEVICE;
}

void *encode_tiled_fn()
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_tried) {
        g_encode_tried = true;
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = fn;
        else
            cudaGetLastError();
    }
    return g_encode_tiled;
}

bool overlaps(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes)
{
    if (!a || !b || a_bytes <= 0 || b_bytes <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)b_bytes && b0 < a0 + (uintptr_t)a_bytes;
}

constexpr int64_t kMaxDim = 0x7fffffff;

// Checks shared by both entry points. Returns GEMM_OK and sets *nothing_to_do
// when M or N is zero.
int check_common(int64_t M, int64_t N, int64_t K, const void *A, const void *B, const void *C,
                 int64_t elem, bool *nothing_to_do)
{
    *nothing_to_do = false;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) {
        *nothing_to_do = true;
        return GEMM_OK;
    }
    if (!C)
        return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B))
        return GEMM_ERR_INVALID_ARG;
    if (M * N > (int64_t)1 << 52 || M * K > (int64_t)1 << 52 || K * N > (int64_t)1 << 52)
        return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (overlaps(C, M * N * 4, A, M * K * elem) || overlaps(C, M * N * 4, B, K * N * elem)))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

int finish(cudaError_t e)
{
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

// Bytes of a copy of a rows x cols matrix of 2-byte values with every row
// padded to a multiple of 8 values (16 bytes), rounded up to 256 bytes.
int64_t padded_copy_bytes(int64_t rows, int64_t cols)
{
    return (rows * ((cols + 7) / 8 * 8) * 2 + 255) / 256 * 256;
}

// The register-tiled fp32 product, K split over cluster CTAs when
// cluster.splits > 1; otherwise, for products with more tiles than SMs, the
// ragged last wave may be split over clusters (sgemm_tail_plan). Unsplit
// 128 x 128 tiles run on the TMA-fed kernel where the operands allow it.
cudaError_t run_f32_tiles(int M, int N, int K, const float *A, const float *B, float *C,
                          const rtm::SplitK &cluster, const DeviceInfo &d, cudaStream_t s,
                          const rtm::SimtTma *prepared = nullptr)
{
    rtm::SimtTma tma;
    tma.encode_tiled = encode_tiled_fn();
    tma.err = d.err;
    tma.wait_limit_ns = kDefaultWaitLimitNs;
    if (prepared)
        tma = *prepared;
    return rtm::launch_sgemm_f32_tiles(M, N, K, A, B, C, cluster, d.sms, s,
                                       tma.encode_tiled ? &tma : nullptr);
}

// Bytes of a copy of a rows x cols fp32 matrix with every row padded to a
// multiple of 4 values (16 bytes), rounded up to 256 bytes.
int64_t padded_copy_bytes_f32(int64_t rows, int64_t cols)
{
    return (rows * ((cols + 3) / 4 * 4) * 4 + 255) / 256 * 256;
}

// Scratch a gemm_f32_ws schedule needs for itself: stream-K partial tiles or
// the workspace split's partial products.
int64_t f32_schedule_bytes(const rtm::F32Schedule &f, int64_t M, int64_t N)
{
    if (f.streamk > 0)
        return rtm::sgemm_streamk_workspace_floats((int)M, (int)N, f.streamk) *
               (int64_t)sizeof(float);
    return f.workspace.splits > 1 ? (int64_t)f.workspace.splits * M * N * (int64_t)sizeof(float)
                                  : 0;
}

// Whether gemm_f32_ws may run `f` on re-pitched copies: stream-K, or no
// workspace split and a schedule whose kernels are all TMA-fed (the cp.async
// kernels read A and B with row strides K and N).
bool f32_schedule_takes_copies(const rtm::F32Schedule &f, int M, int N, int K, int sms)
{
    return f.streamk > 0 ||
           (f.workspace.splits <= 1 && rtm::sgemm_tiles_use_tma(M, N, K, f.cluster, sms));
}

bool rows_on_16_bytes(const void *base, int64_t cols)
{
    return cols % 8 == 0 && (reinterpret_cast<uintptr_t>(base) & 15) == 0;
}

// The fp32 product without a workspace: column strips for short, wide
// products (M <= 32, where 128-row tiles would be mostly empty), the
// register-tiled kernel with 128 x 128 tiles otherwise (64 columns for
// N <= 64, 64 rows for M <= 64), with K split over the CTAs of a cluster
// when the product has too few tiles to fill the GPU. K >= 1.
cudaError_t run_f32_plain(int M, int N, int K, const float *A, const float *B, float *C,
                          const DeviceInfo &d, cudaStream_t s)
{
    if (M <= rtm::kShortMaxM)
        return rtm::launch_sgemm_short(M, N, K, A, B, C, rtm::sgemm_short_splits(M, N, K, d.sms),
                                       s);
    return run_f32_tiles(M, N, K, A, B, C, rtm::sgemm_cluster_schedule(M, N, K, d.sms), d, s);
}

// Shared by the bf16 and fp16 entry points. `workspace` (may be null) lets the
// CTA-pair kernel run on re-pitched copies of operands whose rows do not start
// on 16-byte boundaries.
int run_bf16(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, float *C,
             void *stream, uint64_t wait_limit_ns, int mute_producer, int f16 = 0,
             void *workspace = nullptr, int64_t workspace_bytes = 0)
{
    bool nothing = false;
    int st = check_common(M, N, K, A, B, C, 2, &nothing);
    if (st != GEMM_OK || nothing)
        return st;
    if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace))
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 1) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 1) != 0)))
        return GEMM_ERR_ALIGNMENT;
    // Rows on 16-byte boundaries (the TMA stride rule) take the TMA kernels;
    // anything else the kernels with load-and-swizzle producer warps (CTA
    // pairs for M > 128, the transposed product for M <= 128), unless a
    // workspace allows re-pitched copies for the CTA-pair TMA kernel.
    const bool a_rows16 = rows_on_16_bytes(A, K);
    const bool b_rows16 = rows_on_16_bytes(B, N);
    const bool c_rows16 = rows_on_16_bytes(C, N);
    const bool tma_ok = a_rows16 && b_rows16 && c_rows16;
    DeviceInfo d;
    st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return finish(rtm::launch_zero_fill(C, M * N, s));
    rtm::TcLaunch L;
    L.M = (int)M;
    L.N = (int)N;
    L.K = (int)K;
    L.A = A;
    L.B = B;
    L.C = C;
    L.err = d.err;
    L.wait_limit_ns = wait_limit_ns;
    L.mute_producer = mute_producer;
    L.sm_count = d.sms;
    L.f16 = f16;
    L.encode_tiled = encode_tiled_fn();
    if (!L.encode_tiled)
        return GEMM_ERR_LAUNCH;
    if (M > 128) {
        // CTA pairs (256-row tiles). C needs only 4-byte alignment there; A
        // and B rows must start on 16-byte boundaries, directly or in copies.
        const int64_t need = (a_rows16 ? 0 : padded_copy_bytes(M, K)) +
                             (b_rows16 ? 0 : padded_copy_bytes(K, N));
        // Tall and narrow (N <= 128) with long K: A streams through 128-row
        // tiles with K split over a cluster, as for short, wide products. At
        // 128 < N <= 256 the CTA pairs (one 256-wide tile column, K split in
        // two when the tiles leave pairs idle) measured faster on GB300:
        // 8192 x 256 x 8192 43.1 -> 36.4 us, 16384 x 256 x 4096 53.2 -> 34.9 us.
        const int64_t s_tiles = (M + 127) / 128 * ((N + rtm::tcs_cols((int)N) - 1) / rtm::tcs_cols((int)N));
        const int s_splits = rtm::long_k_splits(s_tiles, K, d.sms);
        if (need == 0 && N <= 128 && s_splits > 0)
            return finish(rtm::launch_gemm_tc_t(L, s_splits, false, s));
        if (need == 0)
            return finish(rtm::launch_gemm_tc_pair(L, s));
        // Tall and narrow with long K on rows off 16-byte boundaries: the
        // tiling above with producer warps in place of TMA, with or without a
        // workspace (a 256-wide pair tile would be mostly zero fill; on GB300,
        // 4097 x 100 x 8190: pairs 108 us, re-pitch + TMA pairs 55 us, this
        // 33 us; 8192 x 62 x 4094: 58, 54, 27 us).
        if (N <= 128 && s_splits > 0)
            return finish(rtm::launch_gemm_tc_any_t(L, s_splits, false, s));
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        if (ws && (reinterpret_cast<uintptr_t>(ws) & 15) == 0 && workspace_bytes >= need) {
            if (overlaps(ws, need, A, M * K * 2) || overlaps(ws, need, B, K * N * 2) ||
                overlaps(ws, need, C, M * N * 4))
                return GEMM_ERR_INVALID_ARG;
            if (!a_rows16) {
                uint16_t *a_copy = reinterpret_cast<uint16_t *>(ws);
                const int64_t lda = (K + 7) / 8 * 8;
                cudaError_t e = rtm::launch_pack_rows_2b(A, M, K, a_copy, lda, d.sms, s);
                if (e != cudaSuccess)
                    return finish(e);
                L.A = a_copy;
                L.lda = lda;
                ws += padded_copy_bytes(M, K);
            }
            if (!b_rows16) {
                uint16_t *b_copy = reinterpret_cast<uint16_t *>(ws);
                const int64_t ldb = (N + 7) / 8 * 8;
                cudaError_t e = rtm::launch_pack_rows_2b(B, K, N, b_copy, ldb, d.sms, s);
                if (e != cudaSuccess)
                    return finish(e);
                L.B = b_copy;
                L.ldb = ldb;
            }
            return finish(rtm::launch_gemm_tc_pair(L, s));
        }
        return finish(rtm::launch_gemm_tc_any_pair(L, s));
    }
    // Long K with at most one 128-column tile per SM: the product streams B
    // and is bound by how much of it is in flight, so compute C^T = B^T.A^T
    // (B fills the MMA's 128-row side) and split K over up to 8 CTAs of a
    // cluster (1..128 x 8192 x 8192: 41-56 us before, 27-33 us; 64 x 1024 x
    // 8192: 39.7 -> 14.5 us). That kernel stores C one float at a time, so C
    // rows need no 16-byte alignment there.
    const int64_t t_tiles = (N + 127) / 128;
    const int t_splits = rtm::long_k_splits(t_tiles, K, d.sms);
    if (t_splits > 0 && a_rows16 && b_rows16)
        return finish(rtm::launch_gemm_tc_t(L, t_splits, true, s));
    // A or B rows off 16-byte boundaries: the transposed kernel with producer
    // warps in place of TMA, with the same K-split; without one (short K, or
    // more column tiles than SMs) one CTA per tile, in waves where the tiles
    // outnumber the SMs. That measured faster than persistent 128 x 256 tiles
    // at every width (32 x 20002 x 8190: 228 -> 138 us; 64 x 24002 x 4094:
    // 129 -> 88 us; 1 x 40001 x 1001: 70 -> 47 us).
    if (!tma_ok)
        return finish(rtm::launch_gemm_tc_any_t(L, t_splits > 0 ? t_splits : 1, true, s));
    // One CTA per 128 x BN tile. With M <= 128 there is one row of tiles, so
    // the widest BN that still gives 60 % of the SMs a tile is used (a sweep
    // of BN 256/128/64 over N = 1K..32K, K = 1K..8K on GB300 found it within
    // 1 % of the best width; 128 x 8192 x 8192: 56.0 us at BN 256, 41.5 at 64),
    // but with at most 16 CTAs per row of A: every CTA reads all of A, and
    // more CTAs on one 128-byte line per K-slice queue at its L2 slice
    // (x 8192 x 8192 at BN 64: M = 1 63.1 us, against 52.6 at BN 256;
    // M = 4 53.6 us; M = 8 and up 42 us).
    int bn = 64;
    for (int w : {256, 128}) {
        if ((N + w - 1) / w * 10 >= (int64_t)d.sms * 6) {
            bn = w;
            break;
        }
    }
    while (bn < 256 && (N + bn - 1) / bn > 16 * M)
        bn *= 2;
    return finish(rtm::launch_gemm_bf16_tc_bn(L, bn, s));
}

} // namespace

namespace rtm {
int check_f32_args(int64_t M, int64_t N, int64_t K, const float *A, const float *B, const float *C,
                   bool *nothing_to_do)
{
    const int st = check_common(M, N, K, A, B, C, 4, nothing_to_do);
    if (st != GEMM_OK || *nothing_to_do)
        return st;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 3) != 0)))
        return GEMM_ERR_ALIGNMENT;
    return GEMM_OK;
}

cudaError_t launch_zero_fill(float *C, int64_t count, cudaStream_t stream)
{
    if (count <= 0)
        return cudaSuccess;
    const bool vec = count % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    const int64_t items = vec ? count / 4 : count;
    int64_t blocks = (items + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    if (vec)
        zero_fill4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<float4 *>(C),
                                                                items);
    else
        zero_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(C, count);
    return cudaGetLastError();
}
} // namespace rtm

extern "C" {

int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, const float *B, float *C,
             void *stream)
{
    bool nothing = false;
    int st = check_common(M, N, K, A, B, C, 4, &nothing);
    if (st != GEMM_OK || nothing)
        return st;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 3) != 0)))
        return GEMM_ERR_ALIGNMENT;
    DeviceInfo d;
    st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return finish(rtm::launch_zero_fill(C, M * N, s));
    return finish(run_f32_plain((int)M, (int)N, (int)K, A, B, C, d, s));
}

int gemm_f32_schedule(int64_t M, int64_t N, int64_t K, int use_workspace, int *kind, int *splits)
{
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim ||
        M * N > (int64_t)1 << 52 || M * K > (int64_t)1 << 52 || K * N > (int64_t)1 << 52)
        return GEMM_ERR_INVALID_ARG;
    int k = GEMM_F32_NO_KERNEL, s = 1;
    if (M > 0 && N > 0 && K > 0) {
        DeviceInfo d;
        const int st = current_device(&d);
        if (st != GEMM_OK)
            return st;
        if (M <= rtm::kShortMaxM) {
            k = GEMM_F32_COLUMN_STRIPS;
            s = rtm::sgemm_short_splits((int)M, (int)N, (int)K, d.sms);
        } else {
            rtm::SplitK cluster;
            if (use_workspace) {
                const rtm::F32Schedule f = rtm::sgemm_ws_schedule((int)M, (int)N, (int)K, d.sms);
                cluster = f.cluster;
                if (f.streamk > 0) {
                    k = GEMM_F32_TILES_STREAM_K;
                    s = f.streamk;
                } else if (f.workspace.splits > 1) {
                    k = GEMM_F32_TILES_WORKSPACE;
                    s = f.workspace.splits;
                }
            } else {
                cluster = rtm::sgemm_cluster_schedule((int)M, (int)N, (int)K, d.sms);
            }
            if (k == GEMM_F32_NO_KERNEL && cluster.tile.m == rtm::simt_tiles::kTallTileM) {
                k = cluster.splits > 1 ? GEMM_F32_TALL_TILES_CLUSTER : GEMM_F32_TALL_TILES;
                s = cluster.splits;
            }
            if (k == GEMM_F32_NO_KERNEL && cluster.tile.n == rtm::simt_tiles::kWideTileN) {
                k = cluster.splits > 1 ? GEMM_F32_WIDE_TILES_CLUSTER : GEMM_F32_WIDE_TILES;
                s = cluster.splits;
            }
            if (k == GEMM_F32_NO_KERNEL) {
                k = cluster.splits > 1 ? GEMM_F32_TILES_CLUSTER : GEMM_F32_TILES;
                s = cluster.splits;
                if (cluster.splits <= 1) {
                    const rtm::TailPlan tail = rtm::sgemm_tail_plan((int)M, (int)N, (int)K, d.sms);
                    if (tail.tail.splits > 1) {
                        k = GEMM_F32_TILES_TAIL_CLUSTER;
                        s = tail.tail.splits;
                    }
                }
            }
        }
    }
    if (kind)
        *kind = k;
    if (splits)
        *splits = s;
    return GEMM_OK;
}

int64_t gemm_f32_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim ||
        M * N > (int64_t)1 << 52 || M * K > (int64_t)1 << 52 || K * N > (int64_t)1 << 52)
        return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || K == 0)
        return 0;
    DeviceInfo d;
    const int st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    if (M <= rtm::kShortMaxM)
        return 0;  // short, wide products split K without a workspace
    const rtm::F32Schedule f = rtm::sgemm_ws_schedule((int)M, (int)N, (int)K, d.sms);
    int64_t copies = 0;  // rows the shape puts off 16-byte boundaries, re-pitched
    if (f32_schedule_takes_copies(f, (int)M, (int)N, (int)K, d.sms))
        copies = (K % 4 ? padded_copy_bytes_f32(M, K) : 0) + (N % 4 ? padded_copy_bytes_f32(K, N) : 0);
    return copies + f32_schedule_bytes(f, M, N);
}

int gemm_f32_ws(int64_t M, int64_t N, int64_t K, const float *A, const float *B, float *C,
                void *workspace, int64_t workspace_bytes, void *stream)
{
    bool nothing = false;
    int st = check_common(M, N, K, A, B, C, 4, &nothing);
    if (st != GEMM_OK || nothing)
        return st;
    if (workspace_bytes < 0 || (workspace_bytes > 0 && !workspace))
        return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (reinterpret_cast<uintptr_t>(workspace) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 3) != 0)))
        return GEMM_ERR_ALIGNMENT;
    DeviceInfo d;
    st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return finish(rtm::launch_zero_fill(C, M * N, s));
    if (M <= rtm::kShortMaxM)
        return finish(run_f32_plain((int)M, (int)N, (int)K, A, B, C, d, s));
    const rtm::F32Schedule f = rtm::sgemm_ws_schedule((int)M, (int)N, (int)K, d.sms);
    rtm::SimtTma tma;
    tma.encode_tiled = encode_tiled_fn();
    tma.err = d.err;
    tma.wait_limit_ns = kDefaultWaitLimitNs;
    // Operands whose rows are off 16-byte boundaries are first re-pitched into
    // the front of the workspace (rows padded to a multiple of 4 values), when
    // the schedule then runs on TMA-fed kernels only and the workspace holds
    // the copies beside the schedule's own scratch (or, for stream-K, at least
    // the copies: the cluster schedule it falls back to reads them too). The
    // TMA kernels read the copies through their row strides; the sums are the
    // same as on the originals.
    const float *Ar = A, *Br = B;
    uint8_t *scratch = static_cast<uint8_t *>(workspace);
    int64_t scratch_bytes = workspace_bytes;
    const bool a_rows16 = K % 4 == 0 && (reinterpret_cast<uintptr_t>(A) & 15) == 0;
    const bool b_rows16 = N % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15) == 0;
    const int64_t copy_a = a_rows16 ? 0 : padded_copy_bytes_f32(M, K);
    const int64_t copy_b = b_rows16 ? 0 : padded_copy_bytes_f32(K, N);
    const int64_t copies = copy_a + copy_b;
    const int64_t own = f32_schedule_bytes(f, M, N);
    const bool tiles_tma = rtm::sgemm_tiles_use_tma((int)M, (int)N, (int)K, f.cluster, d.sms);
    if (copies > 0 && tma.encode_tiled && (reinterpret_cast<uintptr_t>(workspace) & 15) == 0 &&
        f32_schedule_takes_copies(f, (int)M, (int)N, (int)K, d.sms) &&
        (workspace_bytes >= copies + own || (workspace_bytes >= copies && tiles_tma))) {
        if (overlaps(workspace, copies, A, M * K * 4) || overlaps(workspace, copies, B, K * N * 4) ||
            overlaps(workspace, copies, C, M * N * 4))
            return GEMM_ERR_INVALID_ARG;
        if (copy_a) {
            const int64_t lda = (K + 3) / 4 * 4;
            cudaError_t e = rtm::launch_pack_rows_4b(A, M, K, reinterpret_cast<float *>(scratch), lda,
                                                     d.sms, s);
            if (e != cudaSuccess)
                return finish(e);
            Ar = reinterpret_cast<const float *>(scratch);
            tma.lda = lda;
        }
        if (copy_b) {
            const int64_t ldb = (N + 3) / 4 * 4;
            cudaError_t e = rtm::launch_pack_rows_4b(B, K, N, reinterpret_cast<float *>(scratch + copy_a),
                                                     ldb, d.sms, s);
            if (e != cudaSuccess)
                return finish(e);
            Br = reinterpret_cast<const float *>(scratch + copy_a);
            tma.ldb = ldb;
        }
        scratch += copies;
        scratch_bytes -= copies;
    }
    const bool repitched = Ar != A || Br != B;
    if (f.streamk > 0) {
        // Stream-K needs the TMA-fed kernel (row strides multiples of 4 values,
        // 16-byte aligned A, B and scratch); otherwise gemm_f32's schedule runs.
        if (scratch_bytes >= own && tma.encode_tiled &&
            (reinterpret_cast<uintptr_t>(scratch) & 15) == 0 &&
            rtm::sgemm_tma_eligible((int)M, (int)N, (int)K, Ar, Br, tma.lda, tma.ldb)) {
            if (overlaps(scratch, own, A, M * K * 4) || overlaps(scratch, own, B, K * N * 4) ||
                overlaps(scratch, own, C, M * N * 4))
                return GEMM_ERR_INVALID_ARG;
            return finish(rtm::launch_sgemm_f32_streamk((int)M, (int)N, (int)K, Ar, Br, C, tma,
                                                        f.streamk, f.streamk <= d.sms,
                                                        reinterpret_cast<float *>(scratch), s));
        }
        return finish(run_f32_tiles((int)M, (int)N, (int)K, Ar, Br, C, f.cluster, d, s,
                                    repitched ? &tma : nullptr));
    }
    const rtm::SplitK &plan = f.workspace;
    const int64_t need = own;
    if (need == 0 || scratch_bytes < need)
        return finish(run_f32_tiles((int)M, (int)N, (int)K, Ar, Br, C, f.cluster, d, s,
                                    repitched ? &tma : nullptr));
    // The workspace split runs the cp.async kernels on the operands as given
    // (nothing is re-pitched for it).
    if (overlaps(workspace, need, A, M * K * 4) || overlaps(workspace, need, B, K * N * 4) ||
        overlaps(workspace, need, C, M * N * 4))
        return GEMM_ERR_INVALID_ARG;
    return finish(rtm::launch_sgemm_f32_splitk((int)M, (int)N, (int)K, A, B, C, plan,
                                               static_cast<float *>(workspace), s));
}

int gemm_f32_ladder(int rung, int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                    float *C, void *stream)
{
    if (rung < 0 || rung > 6)
        return GEMM_ERR_INVALID_ARG;
    if (rung == 3)
        return gemm_f32(M, N, K, A, B, C, stream);
    bool nothing = false;
    int st = check_common(M, N, K, A, B, C, 4, &nothing);
    if (st != GEMM_OK || nothing)
        return st;
    if ((reinterpret_cast<uintptr_t>(C) & 3) != 0 ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3) != 0 ||
                   (reinterpret_cast<uintptr_t>(B) & 3) != 0)))
        return GEMM_ERR_ALIGNMENT;
    DeviceInfo d;
    st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return finish(rtm::launch_zero_fill(C, M * N, s));
    const cudaError_t e = rtm::launch_sgemm_ladder(rung, (int)M, (int)N, (int)K, A, B, C, s);
    if (e == cudaErrorInvalidValue)
        return GEMM_ERR_INVALID_ARG;  // grid larger than the launch limits
    return finish(e);
}

int gemm_bf16f32(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, float *C,
                 void *stream)
{
    return run_bf16(M, N, K, A, B, C, stream, kDefaultWaitLimitNs, 0);
}

int gemm_f16f32(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, float *C,
                void *stream)
{
    return run_bf16(M, N, K, A, B, C, stream, kDefaultWaitLimitNs, 0, 1);
}

int64_t gemm_bf16f32_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim ||
        M * N > (int64_t)1 << 52 || M * K > (int64_t)1 << 52 || K * N > (int64_t)1 << 52)
        return GEMM_ERR_INVALID_ARG;
    if (M <= 128 || N == 0 || K == 0)
        return 0;
    return padded_copy_bytes(M, K) + padded_copy_bytes(K, N);
}

int gemm_bf16f32_ws(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                    float *C, void *workspace, int64_t workspace_bytes, void *stream)
{
    return run_bf16(M, N, K, A, B, C, stream, kDefaultWaitLimitNs, 0, 0, workspace,
                    workspace_bytes);
}

int gemm_f16f32_ws(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                   float *C, void *workspace, int64_t workspace_bytes, void *stream)
{
    return run_bf16(M, N, K, A, B, C, stream, kDefaultWaitLimitNs, 0, 1, workspace,
                    workspace_bytes);
}

int gemm_bf16f32_selftest_timeout(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                                  const uint16_t *B, float *C, int64_t wait_limit_ns, void *stream)
{
    if (wait_limit_ns < 1000000 || wait_limit_ns > 10000000000LL)
        return GEMM_ERR_INVALID_ARG;
    if (K == 0)
        return GEMM_ERR_INVALID_ARG;  // the K == 0 product launches no waiting kernel
    return run_bf16(M, N, K, A, B, C, stream, (uint64_t)wait_limit_ns, 1);
}

int gemm_f32_selftest_timeout(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                              float *C, int64_t wait_limit_ns, void *stream)
{
    if (wait_limit_ns < 1000000 || wait_limit_ns > 10000000000LL)
        return GEMM_ERR_INVALID_ARG;
    bool nothing = false;
    int st = rtm::check_f32_args(M, N, K, A, B, C, &nothing);
    if (st != GEMM_OK)
        return st;
    if (nothing || K == 0 || M <= rtm::kShortMaxM ||
        !rtm::sgemm_tma_eligible((int)M, (int)N, (int)K, A, B))
        return GEMM_ERR_INVALID_ARG;  // the self-test runs TMA-fed kernels only
    DeviceInfo d;
    st = current_device(&d);
    if (st != GEMM_OK)
        return st;
    // gemm_f32's own schedule for the shape, every TMA-fed launch muted; shapes
    // it runs on tiles that have no TMA-fed kernel (64-row or 64 x 64 tiles)
    // are refused.
    const rtm::SplitK plan = rtm::sgemm_cluster_schedule((int)M, (int)N, (int)K, d.sms);
    const rtm::SimtTile t = rtm::simt_resolve_tile(plan.tile, (int)M, (int)N);
    const bool tma_tile = (t.m == rtm::simt_tiles::kTileM && t.n == rtm::simt_tiles::kTileN) ||
                          (t.m == rtm::simt_tiles::kTallTileM && t.n == rtm::simt_tiles::kNarrowN) ||
                          (t.m == rtm::simt_tiles::kShortTileM && t.n == rtm::simt_tiles::kWideTileN);
    if (!tma_tile)
        return GEMM_ERR_INVALID_ARG;
    rtm::SimtTma tma;
    tma.encode_tiled = encode_tiled_fn();
    tma.err = d.err;
    tma.wait_limit_ns = (uint64_t)wait_limit_ns;
    tma.mute = true;
    if (!tma.encode_tiled)
        return GEMM_ERR_LAUNCH;
    return finish(rtm::launch_sgemm_f32_tiles((int)M, (int)N, (int)K, A, B, C, plan, d.sms,
                                              static_cast<cudaStream_t>(stream), &tma));
}

int gemm_get_device_error(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    DeviceInfo d;
    int st = current_device(&d);
    if (st == GEMM_ERR_LAUNCH)
        return st;
    int value = 0;
    const int zero = 0;
    if (cudaMemcpy(&value, d.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d.err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return value;
}

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK:
        return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG:
        return "GEMM_ERR_INVALID_ARG: negative size, null pointer, overlap or size too large";
    case GEMM_ERR_ALIGNMENT:
        return "GEMM_ERR_ALIGNMENT: a pointer is not aligned to its element size (C: 4 bytes, "
               "bf16/fp16 A and B: 2 bytes, fp32 A and B: 4 bytes)";
    case GEMM_ERR_LAUNCH:
        return "GEMM_ERR_LAUNCH: a CUDA runtime call failed";
    case GEMM_ERR_TIMEOUT:
        return "GEMM_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    case GEMM_ERR_DEVICE:
        return "GEMM_ERR_DEVICE: the current device is not compute capability 10.3 (sm_103a)";
    default:
        return "unknown gemm status";
    }
}

} // extern "C"
