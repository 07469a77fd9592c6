"""GPU tests of the TMA-fed SIMT kernel behind gemm_f32.

gemm_f32 runs its unsplit 128 x 128 tiles on the TMA-fed kernel when
K % 4 == 0, N % 4 == 0 and A and B are 16-byte aligned, and on the cp.async
kernel otherwise. Both sum k in the same order with the same FMA, so a B
placed 4 bytes off a 16-byte boundary (which sends the product to the
cp.async kernel) must give the same bits. Each case is also checked against
the oracle (|C - C_oracle| <= 1e-4 * sum_k |A[i][k] B[k][j]|), with a NaN
guard band around C, and the launched kernel is identified by name from the
profiler's kernel records."""

import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import (assert_bit_exact, assert_close_to_oracle, guard_intact, guarded_output,
                          kernel_names)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# Shapes whose gemm_f32 schedule is unsplit 128 x 128 tiles (more tiles than
# SMs, or K too short to split): ragged M, N and K (K not a multiple of the
# 32-deep slice, down to one partial slice); one whose ragged last wave is
# split over clusters after whole waves of plain tiles (2304^2 x 1024); and
# 128 x 128 tiles with K split over clusters of 2, 4 or 8 CTAs (8: one CTA per
# SM, 512 x 384 x 8192; TMA-fed
# cluster kernel; the same chunks added in the same rank order as the
# cp.async kernel's cluster mode).
SHAPES = [(2000, 2004, 100), (1664, 1920, 260), (4100, 1028, 36), (3000, 1000, 8),
          (1500, 2600, 700), (2304, 2304, 1024), (1024, 1024, 1024), (1000, 1000, 1000),
          (300, 3000, 700), (512, 384, 8192)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    rtm.build()
    return rtm.load_library()


def offset_copy(t: torch.Tensor, floats: int = 1) -> torch.Tensor:
    """The same values in a buffer `floats` fp32 elements past a 16-byte boundary."""
    buf = torch.empty(t.numel() + floats, dtype=t.dtype, device=t.device)
    view = buf[floats:].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 16 == 4 * floats % 16
    return view


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tma_kernel_matches_oracle_and_cp_async_bits(M, N, K):
    assert rtm.gemm_f32_schedule(M, N, K)[0] in ("tiles", "tiles+tail-cluster-split",
                                                 "tiles+cluster-split")
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + 7 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    names = kernel_names(lambda: rtm.gemm_f32(Ad, Bd, out=C))
    assert any("simt_tma::" in n for n in names), names
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "f32")
    Bo = offset_copy(Bd)
    names_cp = kernel_names(lambda: rtm.gemm_f32(Ad, Bo))
    assert not any("simt_tma::" in n for n in names_cp), names_cp
    C_cp = rtm.gemm_f32(Ad, Bo)
    torch.cuda.synchronize()
    assert torch.equal(C, C_cp), "TMA-fed and cp.async kernels differ"


def test_tma_kernel_small_integers_bit_exact():
    M, N, K = 2000, 2004, 100
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=11)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    C0, _ = oracle.gemm(A, B)  # every partial sum is an integer below 2^24: exact
    assert_bit_exact(C, C0)


def test_tma_kernel_unaligned_c_rows():
    # C 4 bytes off a 16-byte boundary: the TMA-fed kernel with scalar stores.
    M, N, K = 1664, 1920, 260
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=12)
    Ad, Bd = A.to(DEV), B.to(DEV)
    ref = rtm.gemm_f32(Ad, Bd)
    buf = torch.full((M * N + 1 + 4096,), float("nan"), device=DEV)
    C = buf[1:1 + M * N].view(M, N)
    names = kernel_names(lambda: rtm.gemm_f32(Ad, Bd, out=C))
    assert any("sgemm_tma_kernel" in n for n in names), names
    torch.cuda.synchronize()
    assert torch.equal(C, ref)
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + M * N:]).all()


def test_tma_kernel_repeats_bit_for_bit():
    M, N, K = 1500, 2600, 700
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=13)
    Ad, Bd = A.to(DEV), B.to(DEV)
    first = rtm.gemm_f32(Ad, Bd)
    for _ in range(3):
        assert torch.equal(rtm.gemm_f32(Ad, Bd), first)


# Every schedule gemm_f32 runs on TMA-fed kernels: 128 x 128 tiles plain, split
# over a cluster, or with a split last wave; 256 x 64 and 64 x 256 tiles.
SELFTEST_SHAPES = [(2000, 2004, 100, ("tiles", "tiles+tail-cluster-split")),
                   (1024, 1024, 1024, ("tiles+cluster-split",)),
                   (2048, 2048, 1024, ("tiles+tail-cluster-split",)),
                   (8192, 64, 4096, ("tall-tiles+cluster-split",)),
                   (64, 8192, 4096, ("wide-tiles+cluster-split",)),
                   (32768, 64, 512, ("tall-tiles",))]


@pytest.mark.parametrize("M,N,K,kinds", SELFTEST_SHAPES)
def test_tma_kernel_bounded_wait_gives_up_and_context_survives(M, N, K, kinds):
    """With the loads muted, every CTA's first wait runs out after 50 ms; the
    kernel records a timeout and returns (every thread still reaches every
    barrier, the cluster barriers too), and the next product on the same
    context is correct."""
    assert rtm.gemm_f32_schedule(M, N, K)[0] in kinds
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=31)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty(M, N, device=DEV)
    assert rtm.get_device_error() == 0
    rtm.gemm_f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert rtm.get_device_error() == 0, "reading the error word clears it"
    assert_close_to_oracle(rtm.gemm_f32(Ad, Bd), A, B, "f32", full=M * N * K <= (1 << 31), seed=M)


def test_tma_selftest_with_c_off_16_byte_boundaries():
    # C 4 bytes past a 16-byte boundary: the muted kernels store C with 4-byte
    # stores as the product kernels do; the guard band stays untouched.
    M, N, K = 1024, 1024, 1024
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=32)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf = torch.full((M * N + 4,), float("nan"), device=DEV)
    C = buf[1:1 + M * N].view(M, N)
    rtm.gemm_f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + M * N:]).all()
    assert_close_to_oracle(rtm.gemm_f32(Ad, Bd), A, B, "f32")


@pytest.mark.parametrize("M,N,K", [(64, 64, 99), (16, 4096, 4096), (256, 256, 256)],
                         ids=["rows_off_16_bytes", "column_strips", "small_tiles"])
def test_tma_selftest_rejects_shapes_off_the_tma_path(M, N, K):
    # K % 4 != 0 (cp.async kernel), M <= 32 (column strips), 64 x 64 tiles
    if M > 32 and K % 4 == 0:
        assert rtm.gemm_f32_schedule(M, N, K)[0] in ("tiles+cluster-split", "tiles")
    A = torch.zeros(M, K, device=DEV)
    B = torch.zeros(K, N, device=DEV)
    with pytest.raises(rtm.GemmError):
        rtm.gemm_f32_selftest_timeout(A, B, torch.empty(M, N, device=DEV), 50_000_000)
