"""GPU tests of the transposed load-and-swizzle kernel: gemm_bf16f32 and
gemm_f16f32 with M <= 128 whose A or B rows do not start on 16-byte
boundaries (tcany::tshort::gemm_tc_any_t_kernel), and the same kernel without
the swap for tall, narrow products (M > 128, N <= 128, long K).

The kernel computes C^T = B^T.A^T: a CTA owns 128 columns of C and 32, 64 or
128 rows, K is split over S CTAs of a cluster (the same S as the TMA-fed
transposed kernel), and producer warps stage the operands with 4- or 8-byte
cp.async copies or 2-byte loads through registers. Checked: the kernel that runs, the oracle (|C - C_oracle| <=
1e-3 * sum_k |A[i][k] B[k][j]|, oracle fed the same 16-bit values), a NaN
guard band around C, small integers bit for bit, bit equality with the
TMA-fed transposed kernel on zero-padded copies of the operands (same tiles,
K-ranges, MMA sequence and summation order), and the bounded waits."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import (assert_bit_exact, assert_close_to_oracle, guard_intact,
                          guarded_output, kernel_names)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ANY_T = "gemm_tc_any_t_kernel"
TCT = "gemm_tct_kernel"

# (M, N, K): access width V, rows per CTA MN and the K-split S on 152 SMs.
SHAPES = [(16, 8190, 8190),    # V 2, MN 32, S 2
          (100, 4094, 4100),   # V 2, MN 128, S 4
          (33, 600, 16388),    # V 4, MN 64, S 8
          (1, 1001, 3001),     # V 1, MN 32, S 2
          (97, 130, 4100),     # V 2, MN 128, S 4, ragged column tile
          (64, 258, 2050),     # V 2, MN 64, S 2
          (128, 1002, 998),    # V 2, MN 128, S 1 (short K)
          (40, 300, 77),       # V 1, MN 64, S 1
          (16, 10002, 2050),   # V 2, MN 32, S 1 (79 column tiles)
          (128, 8188, 8188),   # V 4, MN 128, S 2
          (64, 4094, 4094)]    # V 2, MN 64, S 4 (64 K-blocks, like K = 4096)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def ran(fn, name) -> None:
    names = kernel_names(fn)
    assert any(name in n for n in names), names


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_transposed_any_matches_oracle(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M + 5 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    ran(lambda: rtm.gemm_bf16f32(Ad, Bd, out=C), ANY_T)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16", full=M * N * K <= (1 << 31), seed=M + N)


def test_transposed_any_full_size_sampled():
    # 128 x 8190 x 8190 (S = 2): B streams once, rows on 4-byte boundaries.
    M, N, K = 128, 8190, 8190
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=8191)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16", full=False, seed=5)
    again = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C, again), "the cluster's rank-ordered sum is the same on every call"


@pytest.mark.parametrize("M,N,K", [(64, 258, 2050), (16, 1030, 4100), (128, 1002, 998),
                                   (3, 777, 5001)])
def test_transposed_any_small_integers_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + N + K)
    C = rtm.gemm_bf16f32(A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


# Long K, and the padded K and N (multiples of 8) give the same column tiles
# and the same K-split: the aligned copies run the TMA-fed transposed kernel.
@pytest.mark.parametrize("M,N,K", [(16, 8190, 8190), (100, 4094, 4100), (1, 1001, 3001),
                                   (33, 600, 16388), (16, 10002, 2050), (64, 4094, 4094)])
def test_bits_equal_tma_transposed_on_padded_copies(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "bf16", seed=3 * M + N + K)
    K8, N8 = (K + 7) // 8 * 8, (N + 7) // 8 * 8
    Ap = torch.zeros(M, K8, dtype=torch.bfloat16)
    Bp = torch.zeros(K8, N8, dtype=torch.bfloat16)
    Ap[:, :K] = A
    Bp[:K, :N] = B
    Ad, Bd, Apd, Bpd = A.to(DEV), B.to(DEV), Ap.to(DEV), Bp.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    holder = {}
    ran(lambda: holder.setdefault("Cp", rtm.gemm_bf16f32(Apd, Bpd)), TCT)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.equal(C, holder["Cp"][:, :N])


def test_f16_offset_operands_two_byte_access():
    # fp16, A and B 2 bytes past a 16-byte boundary (2-byte accesses), C 4 bytes past.
    M, N, K = 48, 520, 2600
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=54)
    Ab = torch.zeros(M * K + 1, dtype=torch.float16, device=DEV)
    Bb = torch.zeros(K * N + 1, dtype=torch.float16, device=DEV)
    Cb = torch.full((M * N + 1 + 4096,), float("nan"), device=DEV)
    Ab[1:].copy_(A.flatten().to(DEV))
    Bb[1:].copy_(B.flatten().to(DEV))
    lib = rtm.load_library()

    def call():
        st = lib.gemm_f16f32(M, N, K, Ab.data_ptr() + 2, Bb.data_ptr() + 2, Cb.data_ptr() + 4,
                             torch.cuda.current_stream().cuda_stream)
        assert st == 0

    ran(call, ANY_T)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.isnan(Cb[0]) and torch.isnan(Cb[1 + M * N:]).all()
    assert_close_to_oracle(Cb[1:1 + M * N].view(M, N), A, B, "bf16")


def test_c_off_16_byte_boundaries_keeps_the_tma_transposed_kernel():
    # A and B rows on 16-byte boundaries, C 4 bytes past one: the TMA-fed
    # transposed kernel stores C one float at a time and still runs.
    M, N, K = 64, 4096, 4096
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=55)
    Ad, Bd = A.to(DEV), B.to(DEV)
    Cb = torch.full((M * N + 1 + 4096,), float("nan"), device=DEV)
    lib = rtm.load_library()

    def call():
        st = lib.gemm_bf16f32(M, N, K, Ad.data_ptr(), Bd.data_ptr(), Cb.data_ptr() + 4,
                              torch.cuda.current_stream().cuda_stream)
        assert st == 0

    ran(call, TCT)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.isnan(Cb[0]) and torch.isnan(Cb[1 + M * N:]).all()
    assert_close_to_oracle(Cb[1:1 + M * N].view(M, N), A, B, "bf16", full=False, seed=55)


def test_more_column_tiles_than_sms_run_in_waves():
    # 188 column tiles of 128 > 152 SMs: one CTA per tile, no K split, two waves.
    M, N, K = 64, 24002, 98
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=56)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    ran(lambda: rtm.gemm_bf16f32(Ad, Bd, out=C), ANY_T)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16")


def test_more_column_tiles_than_sms_long_k_sampled():
    # 157 column tiles and 128 K-blocks: no K split (the tiles outnumber the SMs).
    M, N, K = 32, 20002, 8190
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=57)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16", full=False, seed=57)


# Tall, narrow products (M > 128, N <= 128) with long K: the same kernel
# without the swap (A on the MMA's 128-row side, B on its N side), the same
# K-split as the TMA-fed kernel without the swap.
TALL = [(8192, 62, 4094),    # V 2, 64 columns, S 2
        (4097, 100, 8190),   # V 2, 128 columns, S 4, ragged M
        (1000, 120, 8196),   # V 4 (A rows on 8-byte boundaries), S 8
        (300, 33, 2049)]     # V 1, 64 columns, S 2


@pytest.mark.parametrize("M,N,K", TALL)
def test_tall_narrow_matches_oracle(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M + 11 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    ran(lambda: rtm.gemm_bf16f32(Ad, Bd, out=C), ANY_T)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "bf16", full=M * N * K <= (1 << 31), seed=M + N)


@pytest.mark.parametrize("M,N,K", TALL)
def test_tall_narrow_bits_equal_tma_kernel_on_padded_copies(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "bf16", seed=5 * M + N + K)
    K8, N8 = (K + 7) // 8 * 8, (N + 7) // 8 * 8
    Ap = torch.zeros(M, K8, dtype=torch.bfloat16)
    Bp = torch.zeros(K8, N8, dtype=torch.bfloat16)
    Ap[:, :K] = A
    Bp[:K, :N] = B
    Ad, Bd, Apd, Bpd = A.to(DEV), B.to(DEV), Ap.to(DEV), Bp.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    holder = {}
    ran(lambda: holder.setdefault("Cp", rtm.gemm_bf16f32(Apd, Bpd)), TCT)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.equal(C, holder["Cp"][:, :N])


def test_tall_narrow_small_integers_bit_exact():
    M, N, K = 1000, 100, 4100
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=58)
    C = rtm.gemm_bf16f32(A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


@pytest.mark.parametrize("M,N,K", [(100, 258, 130), (64, 1030, 4098), (1, 1001, 3001),
                                   (100, 24002, 130), (4097, 100, 8190)],
                         ids=["split1_4byte", "split4_4byte", "split2_2byte", "waves_4byte",
                              "tall_split4_4byte"])
def test_muted_producers_every_wait_gives_up(M, N, K):
    """The producer warps load nothing: the MMA issuer's and the epilogue's
    bounded waits run out after 50 ms, every thread still reaches the cluster
    barriers, the kernel records a timeout and returns, and the next product
    is correct."""
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M + N)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty(M, N, device=DEV)
    assert rtm.get_device_error() == 0
    rtm.gemm_bf16f32_selftest_timeout(Ad, Bd, C, wait_limit_ns=50_000_000)
    assert rtm.get_device_error() == -4
    assert rtm.get_device_error() == 0, "reading the error word clears it"
    C = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")
