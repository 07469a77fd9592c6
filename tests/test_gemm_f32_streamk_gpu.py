"""GPU tests of stream-K in gemm_f32_ws (products with at most one 128 x 128
tile per SM, K % 4 == 0 and N % 4 == 0, 16-byte-aligned operands).

The CTAs take equal ranges of the tiles x K-slices iterations; a tile split
between CTAs has its parts written to the workspace and added by a fixup
kernel in increasing K order. Checked: the schedule the planner reports, the
oracle (|C - C_oracle| <= 1e-4 * sum_k |A[i][k] B[k][j]|), bit-exact repeats
and small integers, a workspace and a C guard band filled with NaN (every
part the fixup reads must have been written by this call), C rows off
16-byte boundaries, and operands the TMA loads cannot take (the call then
runs gemm_f32's schedule)."""

import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_bit_exact, assert_close_to_oracle, guard_intact, guarded_output

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (M, N, K): ragged tiles and K (2052 = 64 slices + 4), tiles split among 2-14
# CTAs, 1-16 tiles per CTA range boundary.
SHAPES = [(1024, 1024, 1024), (512, 512, 8192), (640, 640, 4096), (1000, 1000, 1000),
          (900, 700, 2052), (700, 1300, 8192), (1920, 1000, 1024)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    rtm.build()
    return rtm.load_library()


def workspace_for(M, N, K, fill=float("nan")):
    need = rtm.gemm_f32_workspace_bytes(M, N, K)
    assert need > 0
    return torch.full((need // 4 + 1024,), fill, device=DEV)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_streamk_matches_oracle(M, N, K):
    assert rtm.gemm_f32_schedule(M, N, K, workspace=True)[0] == "tiles+stream-k"
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 3 + N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    ws = workspace_for(M, N, K)  # NaN: a part read but not written would show
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32_ws(Ad, Bd, out=C, workspace=ws)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "f32")
    again = rtm.gemm_f32_ws(Ad, Bd, workspace=ws)
    assert torch.equal(C, again), "stream-K must repeat bit for bit"


def test_streamk_small_integers_bit_exact():
    M, N, K = 900, 700, 2052
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=21)
    C = rtm.gemm_f32_ws(A.to(DEV), B.to(DEV), workspace=workspace_for(M, N, K))
    C0, _ = oracle.gemm(A, B)  # partial sums are integers below 2^24: exact
    assert_bit_exact(C, C0)


def test_streamk_unaligned_c_rows():
    M, N, K = 1000, 1000, 1000
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=22)
    Ad, Bd = A.to(DEV), B.to(DEV)
    ws = workspace_for(M, N, K)
    ref = rtm.gemm_f32_ws(Ad, Bd, workspace=ws)
    buf = torch.full((M * N + 2 + 4096,), float("nan"), device=DEV)
    C = buf[1:1 + M * N].view(M, N)  # 4 bytes past a 16-byte boundary
    rtm.gemm_f32_ws(Ad, Bd, out=C, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(C, ref)
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + M * N:]).all()


def test_streamk_falls_back_when_tma_cannot_load():
    # B 4 bytes past a 16-byte boundary: TMA cannot stage it, so gemm_f32_ws
    # runs gemm_f32's schedule (the cluster split), same result as gemm_f32.
    M, N, K = 1024, 1024, 1024
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=23)
    Ad = A.to(DEV)
    bbuf = torch.empty(K * N + 1, device=DEV)
    Bo = bbuf[1:].view(K, N)
    Bo.copy_(B.to(DEV))
    C = rtm.gemm_f32_ws(Ad, Bo, workspace=workspace_for(M, N, K))
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "f32")
    assert torch.equal(C, rtm.gemm_f32(Ad, Bo))


def test_streamk_needs_its_workspace():
    # A workspace smaller than gemm_f32_workspace_bytes: gemm_f32's schedule.
    M, N, K = 640, 640, 4096
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=24)
    Ad, Bd = A.to(DEV), B.to(DEV)
    small = torch.empty(1024, device=DEV)
    C = rtm.gemm_f32_ws(Ad, Bd, workspace=small)
    torch.cuda.synchronize()
    assert torch.equal(C, rtm.gemm_f32(Ad, Bd))
    assert_close_to_oracle(C, A, B, "f32")
