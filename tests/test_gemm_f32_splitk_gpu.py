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


def _copy_bytes(rows, cols):
    return (rows * ((cols + 3) // 4 * 4) * 4 + 255) // 256 * 256


# Workspace only where the schedule prices a workspace schedule below the split
# over cluster CTAs (which needs none): the workspace split (long K over few
# tiles of 64 rows or columns) or stream-K (few 128 x 128 tiles); and, for a
# schedule on TMA-fed kernels, re-pitched copies of the operands whose rows the
# shape puts off 16-byte boundaries (A for K % 4 != 0, B for N % 4 != 0).
# 8192 x 64 x 4096 (on 256 x 64 tiles) and 256^3 split over clusters, 4096^3
# fills the GPU unsplit: none. 1000 x 1000 x 999 splits over clusters and
# 4097 x 3001 x 1023 splits its last wave over clusters, both on 128 x 128
# tiles: copies only.
@pytest.mark.parametrize("M,N,K,kind", [(48, 2048, 8192, "ws"), (512, 512, 8192, "sk"),
                                        (8192, 64, 4096, None), (2048, 128, 4096, "sk"),
                                        (1024, 1024, 1024, "sk"), (1000, 1000, 999, "copies"),
                                        (256, 256, 256, None), (4096, 4096, 4096, None),
                                        (4097, 3001, 1023, "copies")])
def test_workspace_size_policy(M, N, K, kind):
    n = rtm.gemm_f32_workspace_bytes(M, N, K)
    assert (n > 0) == (kind is not None)
    sched, splits = rtm.gemm_f32_schedule(M, N, K, workspace=True)
    if kind == "copies":
        assert sched in ("tiles+cluster-split", "tiles+tail-cluster-split")
        assert n == (_copy_bytes(M, K) if K % 4 else 0) + (_copy_bytes(K, N) if N % 4 else 0)
    elif kind == "ws":
        assert sched == "tiles+workspace-split"
        assert n % (M * N * 4) == 0 and n // (M * N * 4) == splits and 2 <= splits <= 32
    elif kind == "sk":
        # One 128 x 128 part per (CTA, tile) pair a range boundary cuts.
        assert sched == "tiles+stream-k"
        tiles = ((M + 127) // 128) * ((N + 127) // 128)
        assert n == (tiles + splits - 1) * 128 * 128 * 4


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
