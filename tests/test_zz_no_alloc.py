"""GPU test of gemm_f32_noalloc, the entry point for callers that cannot
allocate device memory (code hosted by an application that owns all device
memory, or that must not fail for lack of memory once loaded): the split-K
product with its workspace built into the library as a fixed 24 MiB array.

Called through the C ABI and compared with gemm_f32_ws (the same product with
a caller-provided workspace) within the fp32 tolerance of the other tests
(|C - C_ref| <= 1e-4 * sum_k |A[i][k] B[k][j]|), on two calls in a row with
different data, so the second call starts from the first call's leftovers in
the shared array. This file is named to be collected last."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads

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


def call_noalloc(f, A, B):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), device=DEV)
    st = f(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == 0, rtm.status_string(st)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("M,N,K", [(512, 512, 8192), (48, 2048, 8192)])
def test_noalloc_matches_workspace_entry_point_two_calls(noalloc, M, N, K):
    need = rtm.gemm_f32_workspace_bytes(M, N, K)
    assert 0 < need <= SCRATCH_BYTES, "the shape uses the built-in scratch"
    for call, seed in enumerate((101, 202)):
        A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=seed + M)
        Ad, Bd = A.to(DEV), B.to(DEV)
        ref = rtm.gemm_f32_ws(Ad, Bd)  # existing entry point, caller workspace
        got = call_noalloc(noalloc, Ad, Bd)
        _, S = oracle.gemm(A, B)
        diff = (got.double() - ref.double()).abs().cpu().numpy()
        assert np.all(np.isfinite(got.cpu().numpy())), f"call {call}: non-finite output"
        assert np.all(diff <= 1e-4 * S), f"call {call}: max diff/S {float((diff / S).max()):.3e}"


def test_noalloc_rejects_products_needing_more_scratch(noalloc):
    M, N, K = 15360, 128, 8192  # 120 tiles: split five ways (37.5 MB) on a 152-SM GPU
    need = rtm.gemm_f32_workspace_bytes(M, N, K)
    if need <= SCRATCH_BYTES:
        pytest.skip("on this GPU the split of this shape fits the built-in scratch")
    A = torch.zeros(M, K, device=DEV)
    B = torch.zeros(K, N, device=DEV)
    C = torch.zeros(M, N, device=DEV)
    st = noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                 torch.cuda.current_stream().cuda_stream)
    assert st == -1  # GEMM_ERR_INVALID_ARG: beyond the fixed 24 MiB
