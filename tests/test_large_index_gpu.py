"""Products whose C has more than 2^31 elements, so that every index computed
in 32 bits would overflow: the register-tiled SIMT kernel, the tensor-core
CTA-pair kernel and the column-strip kernel for short, wide products. C is
about 8.6 GB; the check gathers seeded sample entries (and the last rows and
columns) on the device and compares them with the oracle's sampled product."""

import numpy as np
import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def check_sampled(C, A, B, tol, seed):
    M, N = C.shape
    rows, cols = workloads.sample_indices(M, N, count=4096, seed=seed)
    got = C[rows.to(DEV), cols.to(DEV)].double().cpu().numpy()
    C0, S = oracle.gemm_sampled(A, B, rows, cols)
    assert np.all(np.isfinite(got))
    ratio = np.abs(got - C0) / np.where(S == 0, 1.0, S)
    assert np.all(ratio <= tol), f"worst err/S {float(ratio.max()):.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_c_beyond_2_pow_31_elements(dtype):
    M, N, K = 46341, 46344, 8   # M * N = 2,147,627,304 > 2^31
    assert M * N > 2 ** 31
    A, B = workloads.make_inputs(M, N, K, "uniform", dtype, seed=91)
    C = torch.empty(M, N, device=DEV)
    fn = rtm.gemm_f32 if dtype == "f32" else rtm.gemm_bf16f32
    fn(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    check_sampled(C, A, B, 1e-4 if dtype == "f32" else 1e-3, seed=91)
    del C
    torch.cuda.empty_cache()


def test_short_wide_c_beyond_2_pow_31_elements():
    M, N, K = 9, (1 << 28) - 8, 2   # M * N > 2^31, column-strip kernel
    assert M * N > 2 ** 31
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=92)
    C = torch.empty(M, N, device=DEV)
    rtm.gemm_f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    check_sampled(C, A, B, 1e-4, seed=92)
    del C
    torch.cuda.empty_cache()
