"""GPU parity tests of gemm_bf16f32 (tcgen05 tensor-core kernel) against the
CPU oracle fed the same bf16 values, through the C ABI (ctypes binding)."""

import pytest
import torch

import oracle
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


def run(A, B):
    C = rtm.gemm_bf16f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    return C


def bf16_inputs(M, N, K, dist="normal", seed=0):
    return workloads.make_inputs(M, N, K, dist, "bf16", seed=seed)


def test_full_size_workload_sampled():
    """The 8192^3 bf16 workload, as the bench launches it; 4096+ sampled entries."""
    w = workloads.WORKLOADS["bf16_8192_normal"]
    A, B = workloads.workload_inputs(w)
    C = run(A, B)
    assert_close_to_oracle(C, A, B, "bf16", full=False, seed=w.seed)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 256, 256), (1024, 1024, 1024),
                                   (1000, 1000, 1000), (129, 264, 72), (1, 8, 8), (300, 8, 520),
                                   (2048, 4096, 512), (4097, 3000, 1032)])
def test_parity_shapes(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=M * 3 + N + K)
    C = run(A, B)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(C, A, B, "bf16", full=full, seed=M + N + K)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 136, 1000), (640, 512, 4096),
                                   (1, 8, 8), (257, 264, 8)])
def test_small_integer_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + 2 * N + 3 * K)
    C = run(A.to(torch.bfloat16), B.to(torch.bfloat16))  # {-4..4} is exact in bf16
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_identity_and_permutation_exact():
    g = torch.Generator().manual_seed(41)
    A = torch.randn(384, 256, generator=g).to(torch.bfloat16)
    I256 = torch.eye(256).to(torch.bfloat16)
    assert_bit_exact(run(A, I256), A.float().numpy())
    I384 = torch.eye(384).to(torch.bfloat16)
    assert_bit_exact(run(I384, A), A.float().numpy())
    p = torch.randperm(384, generator=g)
    P = torch.zeros(384, 384)
    P[torch.arange(384), p] = 1.0
    assert_bit_exact(run(P.to(torch.bfloat16), A), A[p].float().numpy())
    q = torch.randperm(256, generator=g)
    Q = torch.zeros(256, 256)
    Q[q, torch.arange(256)] = 1.0
    assert_bit_exact(run(A, Q.to(torch.bfloat16)), A[:, q].float().numpy())


def test_rank_one_closed_form():
    g = torch.Generator().manual_seed(42)
    M, N, K = 300, 264, 1024
    u = torch.randint(-8, 9, (M,), generator=g).float()
    v = torch.randint(-8, 9, (N,), generator=g).float()
    A = u[:, None].expand(M, K).contiguous().to(torch.bfloat16)
    B = v[None, :].expand(K, N).contiguous().to(torch.bfloat16)
    assert_bit_exact(run(A, B), (K * torch.outer(u, v)).numpy())


@pytest.mark.parametrize("M,N,K", [(200, 264, 136), (128, 256, 64), (3, 8, 16)])
def test_guard_band_untouched(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=43)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    rtm.gemm_bf16f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16")


def test_k_zero_writes_zeros():
    C = torch.full((16, 8), 2.0, device=DEV)
    rtm.gemm_bf16f32(torch.empty(16, 0, dtype=torch.bfloat16, device=DEV),
                     torch.empty(0, 8, dtype=torch.bfloat16, device=DEV), out=C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


@pytest.mark.parametrize("M,N,K", [(16, 16, 12), (300, 129, 77), (1, 1, 1), (257, 260, 1000),
                                   (1000, 1000, 999), (130, 257, 65), (4097, 3001, 1023)])
def test_unaligned_shapes_parity(M, N, K):
    """K or N not a multiple of 8: the load-and-swizzle kernel."""
    A, B = bf16_inputs(M, N, K, seed=M + 7 * N + K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=full, seed=K)


@pytest.mark.parametrize("M,N,K", [(129, 33, 1001), (64, 255, 63)])
def test_unaligned_small_integer_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + N + K)
    C = run(A.to(torch.bfloat16), B.to(torch.bfloat16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_offset_pointers_take_the_load_path():
    """A, B, C at 2/2/4-byte offsets (rows aligned, bases not): correct results."""
    M, N, K = 200, 264, 136
    A, B = bf16_inputs(M, N, K, seed=46)
    Ab = torch.zeros(M * K + 1, dtype=torch.bfloat16, device=DEV)
    Bb = torch.zeros(K * N + 1, dtype=torch.bfloat16, device=DEV)
    Cb = torch.full((M * N + 1,), float("nan"), device=DEV)
    Ab[1:] = A.flatten().to(DEV)
    Bb[1:] = B.flatten().to(DEV)
    lib = rtm.load_library()
    st = lib.gemm_bf16f32(M, N, K, Ab.data_ptr() + 2, Bb.data_ptr() + 2, Cb.data_ptr() + 4,
                          torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(Cb[1:].view(M, N), A, B, "bf16")


@pytest.mark.parametrize("M,N,K", [(200, 130, 90), (120, 100, 33)])
def test_unaligned_guard_band(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=47)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    rtm.gemm_bf16f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16")


def test_repeated_calls_identical():
    A, B = bf16_inputs(2048, 2048, 2048, seed=44)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = rtm.gemm_bf16f32(Ad, Bd)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("M,K", [(256, 256), (128, 256), (256, 4096)],
                         ids=["cta_pair", "single_cta", "cta_pair_k_split"])
def test_bounded_wait_gives_up_and_context_survives(M, K):
    """With the loads muted, every wait runs out after 50 ms; the kernel records
    a timeout and returns, and the next product on the same context is correct.
    M = 256 runs the CTA-pair kernel (with K = 4096 split in two), M = 128 the
    single-CTA kernel."""
    A, B = bf16_inputs(M, 512, K, seed=45)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty(M, 512, device=DEV)
    assert rtm.get_device_error() == 0
    rtm.gemm_bf16f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert rtm.get_device_error() == 0, "reading the error word clears it"
    C = run(A, B)
    assert_close_to_oracle(C, A, B, "bf16")


@pytest.mark.parametrize("M,N,K", [(128, 1024, 512), (100, 264, 1000), (129, 256, 64),
                                   (257, 520, 128)])
def test_single_cta_and_pair_boundary(M, N, K):
    """M <= 128 runs the single-CTA kernel, M > 128 the CTA pair: both near the switch."""
    A, B = bf16_inputs(M, N, K, seed=M * N)
    assert_close_to_oracle(run(A, B), A, B, "bf16")


@pytest.mark.parametrize("M,N,K", [(128, 2048, 1024), (1, 8192, 512), (2, 8192, 256),
                                   (77, 16384, 256), (128, 32768, 128), (16, 2056, 520)])
def test_short_wide_tile_widths(M, N, K):
    """M <= 128: the single-CTA kernel with 128 x 64, 128 x 128 or 128 x 256
    tiles depending on N and M (64, 256, 256, 128, 256 and 64 here on a
    152-SM GPU)."""
    A, B = bf16_inputs(M, N, K, seed=M + N + 3 * K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=full, seed=N)


@pytest.mark.parametrize("M,N,K", [(100, 2056, 136), (128, 16392, 64)])
def test_short_wide_guard_band(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=48)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    rtm.gemm_bf16f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16", full=M * N * K <= (1 << 31), seed=K)


# M <= 128, K of 32 64-deep blocks or more, at most one 128-column tile per SM:
# C^T = B^T.A^T on the tensor cores, K split over S CTAs of a cluster (S for a
# 152-SM GPU noted).
@pytest.mark.parametrize("M,N,K", [(1, 8192, 4096),      # S = 2
                                   (8, 1024, 8192),      # S = 8
                                   (33, 4096, 2048),     # S = 2
                                   (64, 2056, 2048),     # S = 2, ragged N
                                   (100, 1000, 8200),    # S = 8, ragged N and K
                                   (128, 8192, 2048),    # S = 2
                                   (97, 19456, 2048),    # S = 1, 152 tiles
                                   (64, 2048, 8192)])    # 16 tiles: S = 8 only if 16 clusters of 8 fit
def test_transposed_short_wide(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=M * 13 + N + K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=full, seed=M + K)


def test_transposed_full_size_sampled():
    M, N, K = 128, 8192, 8192
    A, B = bf16_inputs(M, N, K, seed=49)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=False, seed=49)


@pytest.mark.parametrize("M,N,K", [(16, 1024, 4096), (128, 2048, 2048)])
def test_transposed_small_integer_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + N + K)
    C = run(A.to(torch.bfloat16), B.to(torch.bfloat16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_transposed_guard_band_and_repeatability():
    M, N, K = 50, 1000, 4096
    A, B = bf16_inputs(M, N, K, seed=50)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    Ad, Bd = A.to(DEV), B.to(DEV)
    rtm.gemm_bf16f32(Ad, Bd, out=C)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert torch.equal(C, C2), "the cluster's rank-ordered sum is the same on every call"
    assert_close_to_oracle(C, A, B, "bf16")


def test_transposed_f16():
    M, N, K = 32, 2048, 4096
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=51)
    C = rtm.gemm_f16f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")


def test_transposed_bounded_wait_gives_up_and_context_survives():
    """64 x 4096 x 4096 runs the transposed kernel with K split over clusters
    of four CTAs; with the loads muted every CTA's waits run out, every thread
    still reaches both cluster barriers, and the next product is correct."""
    A, B = bf16_inputs(64, 4096, 4096, seed=52)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty(64, 4096, device=DEV)
    assert rtm.get_device_error() == 0
    rtm.gemm_bf16f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=False, seed=52)


# M > 128, N <= 128, K of 32 64-deep blocks or more: A on the MMA's 128-row
# side, B (64 or 128 columns) on its N side, K split over S CTAs of a cluster
# (S for 152 SMs).
# 128 < N <= 256 runs on the CTA pairs (K split in two where the tiles leave
# pairs idle); those shapes stay here as the neighbouring case.
@pytest.mark.parametrize("M,N,K", [(8192, 64, 4096),    # S = 2
                                   (4096, 100, 8192),   # S = 4, ragged N, scalar C rows
                                   (2000, 128, 2048),   # S = 2, 128 columns
                                   (300, 8, 4096),      # S = 4
                                   (19456, 120, 2048),  # S = 1, 152 tiles
                                   (1000, 104, 8200),   # S = 8, ragged K
                                   (2048, 64, 8192),    # 16 tiles: S = 8 only if they all fit
                                   (2000, 256, 2048),   # CTA pairs, 256 columns
                                   (19456, 200, 2048),  # CTA pairs, ragged N
                                   (1000, 136, 8200)])  # CTA pairs, K split in two, ragged K
def test_tall_narrow(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=M + 5 * N + K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=full, seed=N + K)


def test_tall_narrow_small_integer_bit_exact():
    A, B = workloads.make_inputs(1024, 64, 4096, "int", "f32", seed=53)
    C = run(A.to(torch.bfloat16), B.to(torch.bfloat16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_tall_narrow_guard_band_and_repeatability():
    M, N, K = 500, 72, 4096
    A, B = bf16_inputs(M, N, K, seed=54)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    Ad, Bd = A.to(DEV), B.to(DEV)
    rtm.gemm_bf16f32(Ad, Bd, out=C)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert torch.equal(C, C2)
    assert_close_to_oracle(C, A, B, "bf16")


def test_tall_narrow_bounded_wait_gives_up_and_context_survives():
    A, B = bf16_inputs(2048, 128, 4096, seed=55)  # clusters of four CTAs
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty(2048, 128, device=DEV)
    assert rtm.get_device_error() == 0
    rtm.gemm_bf16f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=False, seed=55)


# CTA pairs with K split in two: products whose 256 x 256 tiles fill at most
# half the pairs, with K >= 4096 and C rows on 16-byte boundaries. C is
# zero-filled, then each K half adds its tile into C with TMA reduce-adds.
@pytest.mark.parametrize("M,N,K", [(256, 8192, 4096), (130, 264, 4096), (300, 1000, 4104),
                                   (640, 512, 8192), (512, 2048, 4160)])
def test_pair_k_split_parity(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=M + N * 3 + K)
    C = run(A, B)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(C, A, B, "bf16", full=full, seed=M + K)


def test_pair_k_split_small_integer_bit_exact():
    M, N, K = 384, 520, 4096
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=46)
    C = run(A.to(torch.bfloat16), B.to(torch.bfloat16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_pair_k_split_guard_band_and_repeatability():
    """The reduce-adds stay inside C, and the two halves' sum repeats exactly."""
    M, N, K = 300, 1000, 4104
    A, B = bf16_inputs(M, N, K, seed=47)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_bf16f32(Ad, Bd, out=C)
    C2 = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N), "a reduce-add landed outside C"
    assert torch.equal(C, C2)
    assert_close_to_oracle(C, A, B, "bf16")


def test_pair_k_split_f16_and_workspace_path():
    """fp16 operands, and operands re-pitched into a workspace (K, N not
    multiples of 8), through the split CTA-pair kernel."""
    M, N, K = 256, 1024, 4096
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=48)
    C = rtm.gemm_f16f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "bf16")
    M, N, K = 300, 132, 4097
    A, B = bf16_inputs(M, N, K, seed=49)
    C = rtm.gemm_bf16f32_ws(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")


# Rows on 8-byte but not 16-byte boundaries (K and N multiples of 4, not both
# of 8): the load-and-swizzle kernel's producers copy 8-byte vectors with
# cp.async, three K-slices in flight.
@pytest.mark.parametrize("M,N,K", [(1000, 1004, 996), (130, 4100, 4100), (4097, 260, 1028),
                                   (64, 12, 4), (300, 132, 76)])
def test_eight_byte_rows_parity(M, N, K):
    A, B = bf16_inputs(M, N, K, seed=M + 5 * N + K)
    C = run(A, B)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(C, A, B, "bf16", full=full, seed=M + N)


def test_eight_byte_rows_small_integer_bit_exact_and_guard_band():
    M, N, K = 520, 132, 4100
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=50)
    Ad, Bd = A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_bf16f32(Ad, Bd, out=C)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_eight_byte_offset_pointers_f16():
    """Operands 8 bytes past a 16-byte boundary (K, N multiples of 8), fp16."""
    M, N, K = 260, 264, 1000
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=51)
    Abuf = torch.zeros(M * K + 4, dtype=torch.float16, device=DEV)
    Bbuf = torch.zeros(K * N + 4, dtype=torch.float16, device=DEV)
    Ad = Abuf[4:4 + M * K].view(M, K)
    Bd = Bbuf[4:4 + K * N].view(K, N)
    Ad.copy_(A.to(DEV))
    Bd.copy_(B.to(DEV))
    C = rtm.gemm_f16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")
