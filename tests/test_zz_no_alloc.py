"""GPU tests of gemm_f32_noalloc, the fp32 entry point that allocates nothing.

It is for callers that cannot allocate device memory: code hosted by an
application that owns all device memory through its own pool and forbids
other allocations, and code that must not be able to fail for lack of memory
once it is loaded. Its split-K scratch is a fixed 24 MiB array built into the
library and shared by every call on a device, so one call starts from the
previous call's leftovers.

Every product is called through the C ABI and checked
  * against the CPU oracle within the fp32 tolerance of the other tests,
    |C - C_oracle| <= 1e-4 * sum_k |A[i][k] B[k][j]| elementwise, and
  * bit for bit against the entry point it stands in for: gemm_f32_ws with a
    caller workspace (same schedule, same fixed-order reduction), or gemm_f32
    where no split runs,
on two calls in a row with different data, after a call that left NaN in the
shared array. This file is named to be collected last."""

import ctypes

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_close_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH_BYTES = 24 << 20


@pytest.fixture(scope="module")
def noalloc():
    rtm.build()
    lib = rtm.load_library()
    f = lib.gemm_f32_noalloc
    f.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 4
    f.restype = ctypes.c_int
    return f


def call_noalloc(f, A, B, C=None, stream=None):
    M, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.full((M, N), float("nan"), device=DEV)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = f(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), s.cuda_stream)
    assert st == 0, rtm.status_string(st)
    return C


def poison_scratch(f, M, N, K):
    """A call with NaN operands of the given shape: every partial it writes
    into the shared array is NaN."""
    A = torch.full((M, K), float("nan"), device=DEV)
    B = torch.full((K, N), float("nan"), device=DEV)
    C = call_noalloc(f, A, B)
    torch.cuda.synchronize()
    assert torch.isnan(C).all()


def check(f, M, N, K, seed, reference):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=seed)
    Ad, Bd = A.to(DEV), B.to(DEV)
    got = call_noalloc(f, Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(got, A, B, "f32")
    ref = reference(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(got, ref), "differs from the entry point it stands in for"


@pytest.mark.parametrize("M,N,K", [(512, 512, 8192), (48, 2048, 8192)])
def test_noalloc_split_k_two_calls_after_nan(noalloc, M, N, K):
    need = rtm.gemm_f32_workspace_bytes(M, N, K)
    assert 0 < need <= SCRATCH_BYTES, "the shape splits K through the built-in array"
    assert rtm.gemm_f32_schedule(M, N, K, workspace=True)[0] in ("tiles+workspace-split",
                                                                  "tiles+stream-k")
    poison_scratch(noalloc, M, N, K)
    for seed in (101 + M, 202 + M):
        check(noalloc, M, N, K, seed, lambda a, b: rtm.gemm_f32_ws(a, b))


def test_noalloc_smaller_split_after_larger(noalloc):
    big, small = (512, 512, 8192), (200, 300, 4096)
    need_big = rtm.gemm_f32_workspace_bytes(*big)
    need_small = rtm.gemm_f32_workspace_bytes(*small)
    assert 0 < need_small < need_big <= SCRATCH_BYTES
    poison_scratch(noalloc, *big)
    check(noalloc, *small, 303, lambda a, b: rtm.gemm_f32_ws(a, b))
    check(noalloc, *big, 304, lambda a, b: rtm.gemm_f32_ws(a, b))
    check(noalloc, *small, 305, lambda a, b: rtm.gemm_f32_ws(a, b))


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 512), (16, 4096, 1024), (300, 257, 129)])
def test_noalloc_without_split_runs_gemm_f32(noalloc, M, N, K):
    # No workspace split for these shapes: enough tiles (2048^2), the column
    # strips of M <= 32, a small product the cluster split prices lower (its
    # rows off 16-byte boundaries are re-pitched into the array for the TMA-fed
    # kernels, which add the same products in the same order).
    assert rtm.gemm_f32_schedule(M, N, K, workspace=True)[0] not in ("tiles+workspace-split",
                                                                      "tiles+stream-k")
    if M > 32 and (N % 4 == 0 and K % 4 == 0):
        assert rtm.gemm_f32_workspace_bytes(M, N, K) == 0
    for seed in (401, 402):
        check(noalloc, M, N, K, seed + M, lambda a, b: rtm.gemm_f32(a, b))


def test_noalloc_split_beyond_the_array_runs_gemm_f32(noalloc):
    M, N, K = 15360, 128, 8192  # 120 tiles: the workspace split needs more than 24 MiB
    need = rtm.gemm_f32_workspace_bytes(M, N, K)
    if need <= SCRATCH_BYTES:
        pytest.skip("on this GPU the split of this shape fits the built-in array")
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=505)
    Ad, Bd = A.to(DEV), B.to(DEV)
    for _ in range(2):
        got = call_noalloc(noalloc, Ad, Bd)
        torch.cuda.synchronize()
        assert rtm.get_device_error() == 0
        assert_close_to_oracle(got, A, B, "f32", full=False, seed=506)
        assert torch.equal(got, rtm.gemm_f32(Ad, Bd))


def test_noalloc_captured_in_a_graph(noalloc):
    M, N, K = 512, 512, 8192
    assert rtm.gemm_f32_workspace_bytes(M, N, K) > 0
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=606)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.full((M, N), float("nan"), device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call_noalloc(noalloc, Ad, Bd, C, side)  # first call on the device: set-up, eager
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = C.clone()
    graph = torch.cuda.CUDAGraph()
    C.fill_(float("nan"))
    with torch.cuda.graph(graph):
        call_noalloc(noalloc, Ad, Bd, C, torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(C, eager)
    # New operands in the captured buffers, replayed again.
    A2, B2 = workloads.make_inputs(M, N, K, "uniform", "f32", seed=607)
    Ad.copy_(A2)
    Bd.copy_(B2)
    C.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A2, B2, "f32")
    assert torch.equal(C, rtm.gemm_f32_ws(Ad, Bd))
