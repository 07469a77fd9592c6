"""GPU parity tests of the ablation ladder (gemm_f32_ladder rungs 0-6) against
the CPU oracle, through the C ABI."""

import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_bit_exact, assert_close_to_oracle, small_int_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def run(rung, A, B):
    C = rtm.gemm_f32_ladder(rung, A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("rung", [0, 1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1000, 1000, 999), (67, 130, 33), (1, 1, 1),
                                   (129, 65, 300)])
def test_ladder_parity(rung, M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + N + K + rung)
    assert_close_to_oracle(run(rung, A, B), A, B, "f32")


@pytest.mark.parametrize("rung", [0, 1, 2, 3, 4, 5, 6])
def test_ladder_small_integer_bit_exact(rung):
    A, B = small_int_inputs(97, 131, 77, seed=5 + rung)
    assert_bit_exact(run(rung, A, B), (A.to(torch.int64) @ B.to(torch.int64)).numpy())


@pytest.mark.parametrize("rung", [0, 1, 2, 4, 5, 6])
def test_ladder_k_zero(rung):
    C = torch.full((9, 7), 1.0, device=DEV)
    rtm.gemm_f32_ladder(rung, torch.empty(9, 0, device=DEV), torch.empty(0, 7, device=DEV), out=C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


def test_ladder_1024_workload_all_rungs_agree_with_oracle():
    w = workloads.WORKLOADS["f32_1024_uniform"]
    A, B = workloads.workload_inputs(w)
    C0, S = oracle.gemm(A, B)
    for rung in range(7):
        assert_close_to_oracle(run(rung, A, B), A, B, "f32")
