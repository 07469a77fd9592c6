"""GPU tests of the split-K schedule (gemm_f32_ws with a workspace) against
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


def run_ws(A, B):
    C = rtm.gemm_f32_ws(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    return C


# Workspace only where the schedule prices the workspace split below the split
# over cluster CTAs (which needs none): long K over few tiles. 1024^3,
# 1000 x 1000 x 999, 256^3 and 8192 x 64 x 4096 (on 256 x 64 tiles) split over
# clusters; 4096^3 and 4097 x 3001 x 1023 fill the GPU unsplit.
@pytest.mark.parametrize("M,N,K,split", [(48, 2048, 8192, True), (512, 512, 8192, True),
                                         (8192, 64, 4096, False),
                                         (2048, 128, 4096, True), (1024, 1024, 1024, False),
                                         (1000, 1000, 999, False), (256, 256, 256, False),
                                         (4096, 4096, 4096, False), (4097, 3001, 1023, False)])
def test_workspace_size_policy(M, N, K, split):
    n = rtm.gemm_f32_workspace_bytes(M, N, K)
    assert (n > 0) == split
    if split:
        assert n % (M * N * 4) == 0 and 2 <= n // (M * N * 4) <= 32


@pytest.mark.parametrize("name", ["f32_8192x64x4096", "f32_1024_uniform", "f32_1000x1000x999",
                                  "f32_256_uniform"])
def test_split_workloads_parity(name):
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_inputs(w)
    assert_close_to_oracle(run_ws(A, B), A, B, "f32", full=True)


@pytest.mark.parametrize("M,N,K", [(300, 200, 4096), (129, 65, 4000), (64, 8, 4096), (512, 36, 2049)])
def test_split_ragged_parity(M, N, K):
    assert rtm.gemm_f32_workspace_bytes(M, N, K) > 0
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * N + K)
    assert_close_to_oracle(run_ws(A, B), A, B, "f32")


def test_split_small_integer_bit_exact():
    A, B = small_int_inputs(300, 201, 3000, seed=77)
    assert rtm.gemm_f32_workspace_bytes(300, 201, 3000) > 0
    assert_bit_exact(run_ws(A, B), (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_split_is_deterministic():
    A, B = workloads.make_inputs(1024, 512, 2048, "normal", "f32", seed=78)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = rtm.gemm_f32_ws(Ad, Bd)
    C2 = rtm.gemm_f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_small_workspace_falls_back_to_plain_schedule():
    A, B = workloads.make_inputs(512, 64, 2048, "uniform", "f32", seed=79)
    Ad, Bd = A.to(DEV), B.to(DEV)
    small = torch.empty(16, device=DEV)
    C = rtm.gemm_f32_ws(Ad, Bd, workspace=small)
    Cplain = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C, Cplain), "too small a workspace runs gemm_f32's schedule"
    assert_close_to_oracle(C, A, B, "f32")


def test_workspace_overlapping_output_rejected():
    A, B = workloads.make_inputs(256, 64, 2048, "uniform", "f32", seed=80)
    Ad, Bd = A.to(DEV), B.to(DEV)
    need = rtm.gemm_f32_workspace_bytes(256, 64, 2048)
    buf = torch.empty(need // 4 + 256 * 64, device=DEV)
    C = buf[: 256 * 64].view(256, 64)
    with pytest.raises(rtm.GemmError) as e:
        rtm.gemm_f32_ws(Ad, Bd, out=C, workspace=buf)
    assert e.value.status == -1


@pytest.mark.parametrize("N", [8, 63, 64, 65, 128])
def test_split_narrow_tile_boundary(N):
    M, K = 1024, 2048
    assert rtm.gemm_f32_workspace_bytes(M, N, K) > 0
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=N + 5)
    assert_close_to_oracle(run_ws(A, B), A, B, "f32")
