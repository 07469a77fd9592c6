/*
 * register_tiled_matrix_gb300 — dense product C = A.B on one GB300 (sm_103a).
 *
 * C ABI of libgemm_gb300.so. Every entry point takes plain pointers and sizes,
 * returns an int status (gemm_status), never throws, and never allocates
 * device memory per call.
 *
 * The operation. Both entry points compute, for 0 <= i < M and 0 <= j < N,
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * the product that the register-tiling pages build on: one output element
 * is a row of A against a column of B ("【infra之路】理解 Register Tiling",
 * section "先看 Shared Memory 版本里，一个线程在做什么"), computed with three
 * levels of tiling — per-block C tiles over global memory, K-slices staged in
 * shared memory, per-thread (or per-tensor-core) accumulator tiles
 * ("寄存器Tiling跨架构解析", section 1.1; "理解 Register Tiling", sections
 * "Register Tiling 的核心思想" and "关键循环：为什么省了 Shared Memory 读取？").
 * Tiling only re-associates the sum over k, so results agree with the plain
 * definition up to floating-point summation order.
 *
 * Layout. All matrices are dense and row-major with no padding:
 *     A is M x K (element (i,k) at A[i*K + k]),
 *     B is K x N (element (k,j) at B[k*N + j]),
 *     C is M x N (element (i,j) at C[i*N + j]).
 * C is fully overwritten (there is no alpha/beta); entries outside M x N are
 * never written.
 *
 * Ownership and memory. A, B and C are device pointers owned by the caller
 * and must stay valid until the work queued on `stream` has finished. C must
 * not overlap A or B (overlap is detected for the obvious cases and rejected
 * with GEMM_ERR_INVALID_ARG).
 *
 * Streams. `stream` is a cudaStream_t passed as void*; NULL means the legacy
 * default stream. Calls are asynchronous: a GEMM_OK return means the work was
 * queued, not that it finished. The current CUDA device must be the device
 * that owns the pointers and the stream.
 *
 * Degenerate shapes. M == 0 or N == 0: nothing to do, GEMM_OK. K == 0: the
 * empty sum, C is filled with zeros. Negative sizes: GEMM_ERR_INVALID_ARG.
 * A null pointer is an error only when the matrix it names is non-empty.
 *
 * Thread safety. Entry points may be called from several host threads; the
 * only library state is a per-device cache (SM count, driver entry point,
 * kernel attributes) and one device error word per device, both set up on
 * first use.
 *
 * CUDA graphs. After a first call of the same kind on the device (which fills
 * that cache), calls of gemm_f32, gemm_f32_ws, gemm_bf16f32, gemm_f16f32,
 * gemm_bf16f32_ws and gemm_f16f32_ws only enqueue kernels on `stream`: they
 * can be recorded by stream capture and replayed; the pointers, sizes and
 * workspace are fixed at capture. gemm_get_device_error synchronises and
 * must not be called while its stream is being captured.
 */
#ifndef REGISTER_TILED_GEMM_H
#define REGISTER_TILED_GEMM_H

#include <stdint.h>

/* Only the entry points below are exported from the shared library; the
   library is built with hidden default visibility. */
#if defined(__GNUC__) || defined(__clang__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1, /* negative size, null pointer for a non-empty
                                  matrix, C overlapping A or B, size too large */
    GEMM_ERR_ALIGNMENT = -2,   /* a pointer not aligned to its element size
                                  (fp32: 4 bytes, bf16/fp16: 2 bytes; C: 4) */
    GEMM_ERR_LAUNCH = -3,      /* a CUDA runtime call failed (no device, launch
                                  error, earlier sticky error) */
    GEMM_ERR_TIMEOUT = -4,     /* reported by gemm_get_device_error: a bounded
                                  wait inside a kernel gave up */
    GEMM_ERR_DEVICE = -5       /* the current device is not compute capability
                                  10.3 (the library holds sm_103a code only) */
} gemm_status;

/*
 * gemm_f32 — fp32 inputs, fp32 accumulation, fp32 output, on the SIMT FP32
 * pipes with a register micro-tile per thread (the register-tiled kernel:
 * "理解 Register Tiling", sections "Register Tiling 的核心思想" and
 * "关键循环"; "寄存器Tiling跨架构解析", sections 1.1 and 6.1).
 *
 * Any M, N, K >= 0 and any 4-byte-aligned pointers. Each output is a sum of
 * K fp32 products formed with fused multiply-add in an order fixed by the
 * tiling; the error against the exact sum is bounded by a small multiple of
 * K * 2^-24 * sum_k |A[i][k] B[k][j]|. Where the rows of A and B start on
 * 16-byte boundaries (K % 4 == 0, N % 4 == 0, A and B 16-byte aligned) the
 * tensor-memory-access unit stages each K-slice in shared memory (A through
 * a swizzled staging tile that the threads transpose to k-major order);
 * otherwise per-thread asynchronous copies do. Each output's sum runs in the
 * same order either way, so both give the same bits. Products with M <= 32 use a kernel
 * whose threads keep a column strip of C in registers and, where that leaves
 * SMs idle, split K over the CTAs of a cluster, adding the partial sums in a
 * fixed order (results repeat exactly from call to call); no workspace.
 * Larger products with too few C tiles to fill the GPU split K the same way:
 * the 2, 4 or 8 CTAs that share a C tile form a thread-block cluster, park
 * their partial tiles in shared memory and add them through distributed
 * shared memory in rank order. Products with more tiles than SMs may run
 * their whole waves of tiles unsplit and the ragged last wave split that way,
 * as a second launch. gemm_f32_schedule reports the choice.
 */
GEMM_API int gemm_f32(int64_t M, int64_t N, int64_t K,
                      const float *A, const float *B, float *C, void *stream);

/*
 * gemm_f32_schedule — how an M x N x K fp32 product would be computed on the
 * current device: by gemm_f32 when use_workspace == 0, by gemm_f32_ws with a
 * workspace of gemm_f32_workspace_bytes when use_workspace != 0 (also what
 * gemm_f32_noalloc runs when that many bytes are at most its 24 MiB; above
 * that it runs the use_workspace == 0 schedule). Launches nothing. Writes
 * *kind (one of the values below) and *splits (the number of K chunks; 1 when
 * K is not split); either pointer may be null. Returns GEMM_OK, GEMM_ERR_INVALID_ARG for sizes the
 * entry points reject, or GEMM_ERR_LAUNCH / GEMM_ERR_DEVICE when no usable
 * device is current. Products with M == 0, N == 0 or K == 0 report
 * GEMM_F32_NO_KERNEL.
 */
typedef enum gemm_f32_kind {
    GEMM_F32_NO_KERNEL = 0,        /* nothing to multiply (zero fill or no-op) */
    GEMM_F32_TILES = 1,            /* register-tiled kernel, one CTA per C tile */
    GEMM_F32_TILES_CLUSTER = 2,    /* the same, K split over the CTAs of a cluster */
    GEMM_F32_TILES_WORKSPACE = 3,  /* the same, K split through a workspace + reduction */
    GEMM_F32_COLUMN_STRIPS = 4,    /* M <= 32: column strips (K split over a cluster
                                      when splits > 1) */
    GEMM_F32_TILES_TAIL_CLUSTER = 5, /* more tiles than SMs: whole waves of tiles
                                      unsplit, then the ragged last wave with K split
                                      over the CTAs of a cluster (splits = cluster
                                      size) */
    GEMM_F32_TALL_TILES = 6,       /* N <= 64, M > 128: 256 x 64 C tiles (16 x 4 per
                                      thread), one CTA per tile */
    GEMM_F32_TALL_TILES_CLUSTER = 7, /* the same, K split over the CTAs of a cluster.
                                      Both tall kinds fall back to 128 x 64 tiles,
                                      same split, when the rows of B are not on
                                      16-byte boundaries */
    GEMM_F32_WIDE_TILES = 8,       /* 32 < M <= 64, N > 64: 64 x 256 C tiles (4 x 16
                                      per thread), one CTA per tile */
    GEMM_F32_WIDE_TILES_CLUSTER = 9, /* the same, K split over the CTAs of a cluster */
    GEMM_F32_TILES_STREAM_K = 10   /* gemm_f32_ws only: 128 x 128 tiles, the tiles x
                                      K-slices iterations cut into equal ranges over
                                      `splits` CTAs (stream-K); split tiles added by a
                                      second kernel through the workspace */
} gemm_f32_kind;
GEMM_API int gemm_f32_schedule(int64_t M, int64_t N, int64_t K, int use_workspace,
                               int *kind, int *splits);

/*
 * gemm_f32_workspace_bytes — bytes of scratch memory gemm_f32_ws uses for an
 * M x N x K product on the current device, the sum of two parts:
 *   - the schedule's own scratch: 0 when the product has enough C tiles to
 *     fill the GPU, or when splitting K over cluster CTAs (which needs no
 *     workspace, see gemm_f32) is estimated to be at least as fast; otherwise
 *     the size of one of the two workspace schedules below, whichever is
 *     estimated faster: splits * M * N * 4 for the K split, (tiles + ctas - 1)
 *     * 65536 for stream-K (tiles: the product's 128 x 128 C tiles; ctas: the
 *     `splits` gemm_f32_schedule reports);
 *   - when the schedule runs on the kernels that stage K-slices with the
 *     tensor-memory-access unit (stream-K, or 128 x 128, 256 x 64 or 64 x 256
 *     tiles without the K split), room for re-pitched copies of the operands
 *     whose rows the shape puts off 16-byte boundaries: ceil256(M * ceil4(K)
 *     * 4) when K % 4 != 0, ceil256(K * ceil4(N) * 4) when N % 4 != 0.
 * Returns a negative status on invalid sizes (GEMM_ERR_INVALID_ARG) or when
 * no usable device is current (GEMM_ERR_LAUNCH, GEMM_ERR_DEVICE).
 *
 * gemm_f32_ws — the same product as gemm_f32 (same layout, ownership and
 * degenerate-shape rules) for shapes with few C tiles, such as skinny or
 * small products, given a workspace of at least gemm_f32_workspace_bytes(M,
 * N, K) > 0 bytes (device memory owned by the caller, 4-byte aligned, 16-byte
 * aligned for the vector paths, not overlapping A, B or C):
 *   - K split: K is cut into `splits` chunks (a multiple of 32 deep); each
 *     chunk's partial M x N product goes to its own slab of the workspace and
 *     a second kernel adds the slabs into C in increasing chunk order. Up to
 *     32 chunks against a cluster's 8: long K over few tiles.
 *   - stream-K (128 x 128 tiles; K % 4 == 0, N % 4 == 0, A, B and the
 *     workspace 16-byte aligned, else gemm_f32's schedule runs): the product's
 *     tiles x 32-deep K-slices are cut into `splits` equal ranges, one per CTA,
 *     so every SM works the same time; a tile a CTA computes whole goes to C,
 *     parts of tiles shared by several CTAs go to the workspace and a second
 *     kernel adds them in increasing K order.
 * Both give bit-for-bit the same result from call to call. Otherwise (no
 * workspace schedule planned, or the workspace too small) it runs what
 * gemm_f32 runs. Operands whose rows do not start on 16-byte boundaries (K or
 * N not a multiple of 4, or A or B not 16-byte aligned) are first copied into
 * the front of the workspace with rows padded to a multiple of 4 values (A's
 * copy first, B's after it at a 256-byte-rounded offset, the schedule's own
 * scratch after both) when the schedule then runs on tensor-memory-access
 * staging only and the workspace holds the copies beside the schedule's
 * scratch (or, for stream-K, at least the copies, for the cluster schedule it
 * then runs); the copies change no sum, so where gemm_f32 runs the same
 * schedule the results are the same bits. Any other schedule runs on the
 * operands as given. The workspace contents on return are unspecified; two
 * calls in flight at once must not share a workspace. The splits are the
 * pages' global tiling applied to K as well as to C tiles
 * ("寄存器Tiling跨架构解析", sections 1.1 and 2.4: global tiling decides how much
 * work each block gets) and change only the summation order.
 */
GEMM_API int64_t gemm_f32_workspace_bytes(int64_t M, int64_t N, int64_t K);
GEMM_API int gemm_f32_ws(int64_t M, int64_t N, int64_t K,
                         const float *A, const float *B, float *C,
                         void *workspace, int64_t workspace_bytes, void *stream);

/*
 * gemm_f32_noalloc — the gemm_f32_ws product for callers that cannot
 * allocate device memory: code hosted by an application that owns all device
 * memory through its own pool and forbids other allocations, and code that
 * must not be able to fail for lack of memory once loaded. It allocates
 * nothing: the split-K workspace is a fixed 24 MiB array built into the
 * library (every GPU that loads the library holds it until the process
 * exits). The register-tiling pages have no counterpart of this entry point.
 *
 * Same arguments, layout, ownership, degenerate-shape, alignment and error
 * rules as gemm_f32 (argument errors are reported before any CUDA call). It
 * runs what gemm_f32_ws runs with the built-in array as its workspace: the
 * split-K schedule when that split fits in 24 MiB (splits * M * N * 4 bytes,
 * see gemm_f32_workspace_bytes), and otherwise gemm_f32's own schedule, which
 * needs no scratch memory; re-pitched copies of operands whose rows are off
 * 16-byte boundaries where they fit in the array beside that. Every valid
 * product therefore succeeds.
 *
 * The first call on each device looks up the device address of the built-in
 * array (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture. All calls on a device share the array:
 * its contents persist between calls, nothing in it needs to start at zero
 * (a call writes every element of it that it reads, before reading it), and
 * two calls whose work overlaps on the GPU (for example on two streams) race
 * on it.
 */
GEMM_API int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K,
                              const float *A, const float *B, float *C, void *stream);

/*
 * gemm_f32_ladder — the ablation ladder of the register-tiling page: the same
 * fp32 product computed by the kernels the page compares, kept as the page
 * describes them, for measuring what each tiling level buys
 * ("【infra之路】理解 Register Tiling", sections "先看 Shared Memory 版本里，一个
 * 线程在做什么", "Register Tiling 的核心思想", "关键循环", "用一张图对比三个版本").
 *
 *   rung 0  naive: one thread per output, operands read from global memory;
 *   rung 1  shared-memory tiled, TILE = 32, one output per thread
 *           (2 shared reads per output per k);
 *   rung 2  register tiled, 64 x 64 block, 16 x 16 threads, a 4 x 4 block of
 *           outputs per thread (0.5 shared reads per output per k);
 *   rung 3  gemm_f32 itself (8 x 8 per thread, 0.25).
 *
 * Rungs 4-6 are the page's extreme-tile experiment ("寄存器Tiling跨架构解析",
 * section 7.4): rung 2's kernel with only the per-thread tile changed, T x T
 * outputs on the same 16 x 16 threads (a 16T x 16T block, 2/T shared reads
 * per output per k):
 *
 *   rung 4  T = 1 (16 x 16 block);   rung 5  T = 2 (32 x 32 block);
 *   rung 6  T = 8 (128 x 128 block); rung 2 is T = 4.
 *
 * Same layout, ownership, degenerate-shape and error rules as gemm_f32; any
 * shape. GEMM_ERR_INVALID_ARG for a rung outside 0..6, or when M exceeds what
 * the rung's grid can cover (65535 tiles along M: M > 1,048,560 for rungs 0
 * and 4, 2,097,120 for rungs 1 and 5, 4,194,240 for rung 2, 8,388,480 for
 * rung 6).
 */
GEMM_API int gemm_f32_ladder(int rung, int64_t M, int64_t N, int64_t K,
                             const float *A, const float *B, float *C, void *stream);

/*
 * gemm_bf16f32 — bfloat16 inputs, fp32 accumulation and output, on the
 * tcgen05 tensor cores: operands staged in shared memory by TMA, the
 * accumulator tile held in tensor memory (the tensor-core form of the
 * register tile; "寄存器Tiling跨架构解析", sections 2.1 and 6). For M > 128 a
 * cluster of two CTAs computes each 256 x 256 tile with the two-SM MMA
 * (each SM stages half of A and half of B); for M <= 128 one CTA per
 * 128 x 256, 128 x 128 or 128 x 64 tile, or, when K has at least 32 64-deep
 * blocks and the 128-column tiles of C fit on the SMs, the transposed
 * product C^T = B^T.A^T with K split over the CTAs of a cluster (the long
 * operand B on the MMA's 128-row side; the partial sums are added in a fixed
 * order, so results repeat exactly from call to call).
 *
 * A and B hold raw bfloat16 bit patterns (uint16_t), 2-byte aligned; C is
 * 4-byte aligned (else GEMM_ERR_ALIGNMENT). Any M, N, K. When the rows of A
 * and B start on 16-byte boundaries (K % 8 == 0, N % 8 == 0, A and B 16-byte
 * aligned) the operands are staged by the tensor-memory-access unit (C rows
 * may start anywhere 4-byte aligned, except for M <= 128 with fewer than 32
 * K-blocks or more column tiles than SMs, where C must be 16-byte aligned
 * with N % 8 == 0 as well); otherwise by producer warps that copy them 2, 4
 * or 8 bytes at a time into the same swizzled layout (for M > 128 on CTA
 * pairs, or for tall, narrow products, N <= 128 with at least 32 K-blocks, on
 * 128-row tiles with the same K-split as on aligned rows; for M <= 128 on the
 * transposed product, with the same K-split where one applies). This is
 * slower than the TMA staging, with the same
 * arithmetic: for M > 128 the results equal gemm_bf16f32_ws's bit for bit
 * unless that call adds two K halves of a tile, which it may do only when C
 * rows are 16-byte aligned and K >= 4096; for M <= 128 with at least 32
 * K-blocks and at most one 128-column tile per SM they equal, bit for bit,
 * those of the same values zero-padded to rows of a multiple of 8 values.
 * Ragged M, N and K tiles are handled by zero-filled loads and masked stores.
 *
 * Every wait inside the kernel is bounded (a few seconds); if one gives up
 * the kernel records GEMM_ERR_TIMEOUT in the device error word and returns
 * instead of hanging. Read it with gemm_get_device_error.
 */
GEMM_API int gemm_bf16f32(int64_t M, int64_t N, int64_t K,
                          const uint16_t *A, const uint16_t *B, float *C, void *stream);

/*
 * gemm_f16f32 — IEEE half-precision (fp16) inputs, fp32 accumulation and
 * output, on the same tcgen05 kernel as gemm_bf16f32 with the operands'
 * format set to fp16: the pages' own worked example is this HGEMM, fp16 in
 * and fp32 accumulate ("寄存器Tiling跨架构解析", section 6 and 6.1). A and B hold
 * raw fp16 bit patterns; every rule of gemm_bf16f32 applies (alignment,
 * the two staging paths, bounded waits).
 */
GEMM_API int gemm_f16f32(int64_t M, int64_t N, int64_t K,
                         const uint16_t *A, const uint16_t *B, float *C, void *stream);

/*
 * gemm_bf16f32_workspace_bytes — bytes of scratch memory gemm_bf16f32_ws and
 * gemm_f16f32_ws may use for an M x N x K product, whatever the pointers:
 * 0 when M <= 128 or K == 0 or N == 0, otherwise room for a copy of A with
 * rows padded to a multiple of 8 values plus one of B, each rounded up to
 * 256 bytes: ceil256(M * ceil8(K) * 2) + ceil256(K * ceil8(N) * 2). A call
 * uses only the part for the operands it copies (below). Returns
 * GEMM_ERR_INVALID_ARG for negative or oversized dimensions.
 *
 * gemm_bf16f32_ws / gemm_f16f32_ws — the product of gemm_bf16f32 /
 * gemm_f16f32 (same layout, alignment, ownership, degenerate-shape and error
 * rules), fast also when rows do not start on 16-byte boundaries. For M > 128,
 * an operand whose rows are not 16-byte aligned (A when K % 8 != 0 or A is
 * not 16-byte aligned; B likewise with N) is first copied into `workspace`
 * (device memory owned by the caller, 16-byte aligned, not overlapping A, B
 * or C) with its rows padded to 16-byte multiples — A's copy first, B's
 * after it at a 256-byte-rounded offset — and the CTA-pair tensor-core kernel
 * then stages the copies by TMA. The copy is the global level of the pages'
 * tiling adapted to Blackwell, whose tensor-memory-access unit can only start
 * a tile on a 16-byte boundary; the arithmetic is unchanged. When no copy is
 * needed, or the workspace is null, misaligned or smaller than the copies,
 * and for tall, narrow products (N <= 128 with at least 32 K-blocks and the
 * 128-row tiles fitting on the SMs), which the producer warps compute faster
 * than the copies would allow, the call runs exactly what gemm_bf16f32 /
 * gemm_f16f32 runs. The workspace
 * contents on return are unspecified; two calls in flight at once must not
 * share a workspace. A workspace that overlaps A, B or C returns
 * GEMM_ERR_INVALID_ARG.
 */
GEMM_API int64_t gemm_bf16f32_workspace_bytes(int64_t M, int64_t N, int64_t K);
GEMM_API int gemm_bf16f32_ws(int64_t M, int64_t N, int64_t K,
                             const uint16_t *A, const uint16_t *B, float *C,
                             void *workspace, int64_t workspace_bytes, void *stream);
GEMM_API int gemm_f16f32_ws(int64_t M, int64_t N, int64_t K,
                            const uint16_t *A, const uint16_t *B, float *C,
                            void *workspace, int64_t workspace_bytes, void *stream);

/*
 * gemm_get_device_error — synchronises `stream`, then returns and clears the
 * current device's error word: GEMM_OK, or GEMM_ERR_TIMEOUT if a bounded wait
 * in any kernel of this library on this device gave up since the last call.
 * Returns GEMM_ERR_LAUNCH if the synchronisation itself fails.
 */
GEMM_API int gemm_get_device_error(void *stream);

/*
 * gemm_bf16f32_selftest_timeout — failure-detection check for the bounded
 * waits. Launches the gemm_bf16f32 kernel the shape and pointers select (CTA
 * pair for M > 128, single CTA or the transposed K-split kernel otherwise;
 * for rows off 16-byte boundaries the load-and-swizzle kernels) on the given
 * buffers with its producer muted (the tensor-memory-access thread, or the
 * producer warps), so that nothing ever arrives on the stage barriers, and
 * with every wait limited to `wait_limit_ns`. Each waiting warp gives up, the
 * kernel frees its tensor memory, records GEMM_ERR_TIMEOUT in the device
 * error word and returns; the GPU context stays usable. C is left
 * unspecified. Same argument rules as gemm_bf16f32, K > 0, else
 * GEMM_ERR_INVALID_ARG; wait_limit_ns must be in [1e6, 1e10].
 */
GEMM_API int gemm_bf16f32_selftest_timeout(int64_t M, int64_t N, int64_t K,
                                           const uint16_t *A, const uint16_t *B, float *C,
                                           int64_t wait_limit_ns, void *stream);

/*
 * gemm_f32_selftest_timeout — failure-detection check for the bounded waits
 * of gemm_f32's TMA-fed kernels. Runs gemm_f32's schedule for the shape (128
 * x 128 tiles plain, with K split over a cluster or with a split last wave;
 * 256 x 64 or 64 x 256 tiles) on the given buffers with every TMA load muted
 * (each K-slice's bytes are announced on its barrier but never loaded) and
 * every wait limited to `wait_limit_ns`: each CTA's first wait gives up,
 * records GEMM_ERR_TIMEOUT in the device error word and raises the CTA's
 * abort flag; every thread still reaches every barrier (the cluster barriers
 * too) and the kernel returns, leaving the GPU context usable. C is left
 * unspecified. Same argument rules as gemm_f32; the shape must run on those
 * kernels (K > 0, M > 32, K % 4 == 0, N % 4 == 0, A and B 16-byte aligned,
 * not 64-row or 64 x 64 tiles) else GEMM_ERR_INVALID_ARG; wait_limit_ns must
 * be in [1e6, 1e10].
 */
GEMM_API int gemm_f32_selftest_timeout(int64_t M, int64_t N, int64_t K,
                                       const float *A, const float *B, float *C,
                                       int64_t wait_limit_ns, void *stream);

/*
 * gemm_fp32_pipe_peak — measurement of the FP32 FMA pipes that gemm_f32's
 * register tiles feed ("GPU架构基础", the SM and CUDA-core section: the FP32
 * cores of an SM), used as the measured denominator of gemm_f32's roofline.
 * Launches, on `stream`, 4 CTAs of 256 threads per SM, each thread running
 * 16 independent chains of `iters` x 32 dependent FMAs x <- x * a + b on
 * registers only (no memory traffic); with `packed` != 0 the same chains go
 * through the packed two-wide FP32 FMA. Writes the launch's floating-point
 * operation count (2 per FMA) to *flops on the host before returning. The
 * kernel raises clock_out[0] to the largest number of SM clock cycles and
 * clock_out[1] to the largest number of global-timer nanoseconds any CTA
 * spent (atomic maxima; clock_out is a device array of two 8-byte-aligned
 * unsigned 64-bit values that the caller zeroes first), so that
 * clock_out[0] / clock_out[1] is the SM clock in GHz during the run. The
 * caller times the launch (CUDA events on `stream`). Returns
 * GEMM_ERR_INVALID_ARG for iters outside [1, 2^40] or null pointers,
 * GEMM_ERR_ALIGNMENT for a misaligned clock_out, GEMM_ERR_DEVICE when the
 * current device is not sm_103, GEMM_ERR_LAUNCH when the launch fails.
 */
GEMM_API int gemm_fp32_pipe_peak(int64_t iters, int packed, unsigned long long *clock_out,
                                 double *flops, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
GEMM_API const char *gemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* REGISTER_TILED_GEMM_H */
