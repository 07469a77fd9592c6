"""GPU tests of gemm_f32_ws on operands whose rows do not start on 16-byte
boundaries (K % 4 != 0 for A, N % 4 != 0 for B, or offset pointers): the
workspace entry re-pitches them into the front of the workspace (rows padded
to a multiple of 4 values) and runs its schedule on the TMA-fed kernels, which
read the copies through their row strides, when the schedule's kernels are all
TMA-fed (stream-K, or 128 x 128, 256 x 64 or 64 x 256 tiles without a
workspace split).

Checked: the re-pitch and a TMA-fed kernel run, the oracle (|C - C_oracle| <=
1e-4 * sum_k |A[i][k] B[k][j]|), a NaN guard band around C, bit equality with
gemm_f32 (the cp.async kernels on the operands as given) wherever the two run
the same schedule (the TMA-fed and cp.async kernels add the same products in
the same order), repeatability, and that a workspace too small for the
copies runs the operands as given."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_close_to_oracle, guard_intact, guarded_output, kernel_names

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PACK = "pack_rows_kernel"
TMA = ("simt_tma::", "simt_tma_rect::")

# (M, N, K, re-pitched): which operand the shape puts off 16-byte boundaries;
# re-pitched True where the schedule is known to run on TMA-fed kernels (128 x
# 128 tiles or stream-K), None where the planner's tile choice decides.
SHAPES = [(1000, 1000, 999, True),     # A (config 4a)
          (4097, 3001, 1023, True),    # A and B (config 4b)
          (2048, 2046, 1024, True),    # B
          (1000, 1002, 998, True),     # A and B
          (640, 518, 2047, None),      # A and B, few tiles
          (8192, 62, 4093, None),      # A and B, tall, narrow
          (60, 8192, 4093, None)]      # A, short, wide


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def _workspace(M, N, K, extra=0):
    n = rtm.gemm_f32_workspace_bytes(M, N, K)
    return torch.empty(max((n + extra) // 4, 1), device=DEV), n


@pytest.mark.parametrize("M,N,K,repitched", SHAPES)
def test_repitched_operands_match_oracle(M, N, K, repitched):
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=M + 3 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    W, n = _workspace(M, N, K)
    buf, C = guarded_output(M, N, DEV)
    names = kernel_names(lambda: rtm.gemm_f32_ws(Ad, Bd, out=C, workspace=W))
    packed = any(PACK in x for x in names)
    if repitched:
        assert n > 0 and packed, names
    if packed:  # the copies are read only by TMA-fed kernels
        assert any(any(t in x for t in TMA) for x in names), names
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "f32", full=M * N * K <= (1 << 31), seed=M + N)
    again = rtm.gemm_f32_ws(Ad, Bd, workspace=W)
    torch.cuda.synchronize()
    assert torch.equal(C, again), "the same workspace call repeats bit for bit"


@pytest.mark.parametrize("M,N,K,repitched", SHAPES)
def test_bits_equal_gemm_f32_where_the_schedule_is_the_same(M, N, K, repitched):
    kind_ws, splits_ws = rtm.gemm_f32_schedule(M, N, K, workspace=True)
    kind, splits = rtm.gemm_f32_schedule(M, N, K)
    if (kind_ws, splits_ws) != (kind, splits):
        pytest.skip(f"workspace schedule {kind_ws} x{splits_ws} differs from {kind} x{splits}")
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=7 * M + N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    W, _ = _workspace(M, N, K)
    C_ws = rtm.gemm_f32_ws(Ad, Bd, workspace=W)
    C = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.equal(C_ws, C)


def test_full_size_odd_n_sampled():
    # 4096 x 4093 x 4096: B rows on 4-byte boundaries; gemm_f32 runs the
    # cp.async kernel, gemm_f32_ws the TMA-fed one on a re-pitched B.
    M, N, K = 4096, 4093, 4096
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=4093)
    Ad, Bd = A.to(DEV), B.to(DEV)
    W, _ = _workspace(M, N, K)
    C_ws = rtm.gemm_f32_ws(Ad, Bd, workspace=W)
    C = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C_ws, A, B, "f32", full=False, seed=4093)
    if rtm.gemm_f32_schedule(M, N, K, workspace=True) == rtm.gemm_f32_schedule(M, N, K):
        assert torch.equal(C_ws, C)


def test_offset_pointers_are_repitched_with_room():
    # K and N multiples of 4 but A and B 4 bytes past a 16-byte boundary: the
    # shape-only size counts no copies; with room for them beside the
    # schedule's own scratch the call re-pitches both. Both match the oracle.
    M, N, K = 1024, 1024, 1024
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=31)
    Ab = torch.zeros(M * K + 1, device=DEV)
    Bb = torch.zeros(K * N + 1, device=DEV)
    Ab[1:].copy_(A.flatten().to(DEV))
    Bb[1:].copy_(B.flatten().to(DEV))
    Ao, Bo = Ab[1:].view(M, K), Bb[1:].view(K, N)
    W, _ = _workspace(M, N, K)
    C = rtm.gemm_f32_ws(Ao, Bo, workspace=W)
    room = 2 * ((M * ((K + 3) // 4 * 4) * 4 + 255) // 256 * 256)
    W2, _ = _workspace(M, N, K, extra=room)
    names = kernel_names(lambda: rtm.gemm_f32_ws(Ao, Bo, workspace=W2))
    assert any(PACK in x for x in names), names
    C2 = rtm.gemm_f32_ws(Ao, Bo, workspace=W2)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32", full=False, seed=31)
    assert_close_to_oracle(C2, A, B, "f32", full=False, seed=32)


def test_workspace_too_small_for_the_copies_runs_the_operands_as_given():
    M, N, K = 1000, 1000, 999
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=33)
    Ad, Bd = A.to(DEV), B.to(DEV)
    copy_a = (M * ((K + 3) // 4 * 4) * 4 + 255) // 256 * 256
    small = torch.empty((copy_a - 256) // 4, device=DEV)
    names = kernel_names(lambda: rtm.gemm_f32_ws(Ad, Bd, workspace=small))
    assert not any(PACK in x for x in names), names
    C = rtm.gemm_f32_ws(Ad, Bd, workspace=small)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


def test_small_integers_bit_exact():
    M, N, K = 640, 518, 2047
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=34)
    W, _ = _workspace(M, N, K)
    C = rtm.gemm_f32_ws(A.to(DEV), B.to(DEV), workspace=W)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.equal(C.cpu(), (A.to(torch.int64) @ B.to(torch.int64)).to(torch.float32))
