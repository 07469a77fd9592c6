"""GPU parity tests of gemm_bf16f32_ws / gemm_f16f32_ws: operands whose rows do
not start on 16-byte boundaries are re-pitched into the caller's workspace and
multiplied by the CTA-pair tensor-core kernel; checked against the CPU oracle
fed the same 2-byte values, through the C ABI (ctypes binding)."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import (assert_bit_exact, assert_close_to_oracle, guard_intact,
                          guarded_output)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def ws_bytes(M, N, K):
    return rtm.gemm_bf16f32_workspace_bytes(M, N, K)


def pad256(x):
    return (x + 255) // 256 * 256


def copy_bytes(rows, cols):
    return pad256(rows * ((cols + 7) // 8 * 8) * 2)


def run_ws(A, B, dtype="bf16", workspace=None):
    fn = rtm.gemm_bf16f32_ws if dtype == "bf16" else rtm.gemm_f16f32_ws
    C = fn(A.to(DEV), B.to(DEV), workspace=workspace)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    return C


@pytest.mark.parametrize("M,N,K", [
    (300, 129, 77),      # K and N odd
    (257, 264, 1001),    # K odd, N aligned: A re-pitched only
    (384, 259, 512),     # N odd, K aligned: B re-pitched only
    (130, 257, 65),      # one pair tile, both ragged
    (1000, 1000, 999),
    (200, 8, 9),
    (129, 1, 1),
    (640, 33, 4099),
])
def test_parity_unaligned(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M * 5 + N * 3 + K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run_ws(A, B), A, B, "bf16", full=full, seed=K)


@pytest.mark.parametrize("M,N,K", [(4097, 3001, 1023), (8192, 8190, 8190)])
def test_parity_large_sampled(M, N, K):
    """Large ragged shapes, 4096+ sampled entries (the second is the unaligned
    8192-class workload the configs bench times)."""
    w = workloads.WORKLOADS.get("bf16_8192x8190x8190")
    seed = w.seed if (w and (M, N, K) == (w.M, w.N, w.K)) else M + N + K
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=seed)
    assert_close_to_oracle(run_ws(A, B), A, B, "bf16", full=False, seed=seed)


@pytest.mark.parametrize("M,N,K", [(300, 129, 77), (1000, 1000, 999)])
def test_f16_parity(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=M + N + K + 1)
    assert_close_to_oracle(run_ws(A, B, "f16"), A, B, "bf16")


@pytest.mark.parametrize("M,N,K", [(129, 33, 1001), (256, 255, 63), (515, 77, 2047)])
def test_small_integer_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + 2 * N + 3 * K)
    C = run_ws(A.to(torch.bfloat16), B.to(torch.bfloat16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_identity_exact_with_odd_sizes():
    g = torch.Generator().manual_seed(61)
    A = torch.randn(300, 131, generator=g).to(torch.bfloat16)
    I = torch.eye(131).to(torch.bfloat16)
    assert_bit_exact(run_ws(A, I), A.float().numpy())


def test_workspace_size_formula():
    M, N, K = 300, 129, 77
    assert ws_bytes(M, N, K) == copy_bytes(M, K) + copy_bytes(K, N)
    assert ws_bytes(128, N, K) == 0
    assert ws_bytes(M, N, 0) == 0
    assert ws_bytes(M, 0, K) == 0


@pytest.mark.parametrize("M,N,K", [(300, 129, 77), (257, 264, 1001), (384, 259, 512)])
def test_workspace_bounds_and_contents(M, N, K):
    """The call writes nothing past the copies it needs, and whatever the
    workspace held before (NaN here) does not reach C."""
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M + N)
    need = (copy_bytes(M, K) if K % 8 else 0) + (copy_bytes(K, N) if N % 8 else 0)
    ws = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device=DEV)
    ws[:need].view(torch.bfloat16).fill_(float("nan"))
    C = run_ws(A, B, workspace=ws)
    assert bool((ws[need:] == 0xA5).all().item()), "workspace written past the copies"
    assert_close_to_oracle(C, A, B, "bf16")


@pytest.mark.parametrize("M,N,K", [(300, 129, 77), (200, 130, 90)])
def test_guard_band(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M * N)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    rtm.gemm_bf16f32_ws(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16")


def test_offset_pointers():
    """A, B, C at 2/2/4-byte offsets: both operands re-pitched, C stored by rows."""
    M, N, K = 300, 264, 136
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=62)
    Ab = torch.zeros(M * K + 1, dtype=torch.bfloat16, device=DEV)
    Bb = torch.zeros(K * N + 1, dtype=torch.bfloat16, device=DEV)
    Cb = torch.full((M * N + 1,), float("nan"), device=DEV)
    Ab[1:] = A.flatten().to(DEV)
    Bb[1:] = B.flatten().to(DEV)
    ws = torch.empty(ws_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    lib = rtm.load_library()
    st = lib.gemm_bf16f32_ws(M, N, K, Ab.data_ptr() + 2, Bb.data_ptr() + 2, Cb.data_ptr() + 4,
                             ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.isnan(Cb[0]).item()
    assert_close_to_oracle(Cb[1:].view(M, N), A, B, "bf16")


def test_c_offset_only_takes_the_pair_kernel_without_workspace():
    """A and B rows 16-byte aligned, C 4 bytes off: gemm_bf16f32 itself runs the
    CTA-pair kernel with row-by-row C stores (no workspace involved)."""
    M, N, K = 300, 264, 136
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=63)
    Ad, Bd = A.to(DEV), B.to(DEV)  # held until the product has run
    Cb = torch.full((M * N + 2,), float("nan"), device=DEV)
    lib = rtm.load_library()
    st = lib.gemm_bf16f32(M, N, K, Ad.data_ptr(), Bd.data_ptr(),
                          Cb.data_ptr() + 4, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.isnan(Cb[0]).item() and torch.isnan(Cb[-1]).item()
    assert_close_to_oracle(Cb[1:-1].view(M, N), A, B, "bf16")


def test_small_workspace_runs_the_plain_product():
    """Too small a workspace: exactly what gemm_bf16f32 runs (bitwise equal)."""
    M, N, K = 300, 129, 77
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=64)
    Ad, Bd = A.to(DEV), B.to(DEV)
    small = torch.empty(1024, dtype=torch.uint8, device=DEV)
    C1 = rtm.gemm_bf16f32_ws(Ad, Bd, workspace=small)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    assert_close_to_oracle(C1, A, B, "bf16")


def test_m_at_most_128_runs_the_plain_product():
    M, N, K = 128, 129, 77
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=65)
    Ad, Bd = A.to(DEV), B.to(DEV)
    ws = torch.empty(copy_bytes(M, K) + copy_bytes(K, N), dtype=torch.uint8, device=DEV)
    C1 = rtm.gemm_bf16f32_ws(Ad, Bd, workspace=ws)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_workspace_overlapping_c_is_rejected():
    M, N, K = 300, 129, 77
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=66)
    Ad, Bd = A.to(DEV), B.to(DEV)
    big = torch.empty(M * N + ws_bytes(M, N, K) // 4 + 64, device=DEV)
    lib = rtm.load_library()
    st = lib.gemm_bf16f32_ws(M, N, K, Ad.data_ptr(), Bd.data_ptr(),
                             big.data_ptr(), big.data_ptr() + 256, ws_bytes(M, N, K),
                             torch.cuda.current_stream().cuda_stream)
    assert st == -1


def test_repeated_calls_identical():
    A, B = workloads.make_inputs(1000, 1000, 999, "normal", "bf16", seed=67)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = rtm.gemm_bf16f32_ws(Ad, Bd)
    C2 = rtm.gemm_bf16f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
