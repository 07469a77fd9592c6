"""GPU tests of the CTA-pair load-and-swizzle kernel: gemm_bf16f32 and
gemm_f16f32 with M > 128 whose A or B rows do not start on 16-byte boundaries
and no workspace (tcany::pair::gemm_tc_any_pair_kernel).

Each CTA of a pair stages its 128 rows of A and 128 columns of B with 2-, 4-
or 8-byte accesses (the widest that keeps every row aligned) into the swizzled
layout the pair MMA reads. Checked: the kernel that runs, the oracle
(|C - C_oracle| <= 1e-3 * sum_k |A[i][k] B[k][j]|, oracle fed the same 16-bit
values), a NaN guard band around C, small integers bit for bit, and bit
equality with the workspace entry point, which re-pitches the operands and
runs the TMA-fed pair kernel: where that kernel does not split K both issue
the same MMA sequence on the same values."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import (assert_bit_exact, assert_close_to_oracle, guard_intact,
                          guarded_output, kernel_names)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAIR = "gemm_tc_any_pair_kernel"

# Ragged tiles in M, N and K with 2-, 4- and 8-byte accesses; in the last
# row of tiles the odd CTA holds 2 rows (M = 130), none (M = 300, 257) or
# 104 (M = 1000); long K (4100).
SHAPES = [(300, 129, 77), (130, 258, 66), (1000, 1002, 998), (520, 1004, 996),
          (257, 4100, 4100), (1000, 1000, 999), (4097, 3001, 1023)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def pair_ran(fn) -> None:
    names = kernel_names(fn)
    assert any(PAIR in n for n in names), names


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_kernel_matches_oracle(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=M + 3 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    pair_ran(lambda: rtm.gemm_bf16f32(Ad, Bd, out=C))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(C, A, B, "bf16", full=full, seed=M + N)


@pytest.mark.parametrize("M,N,K", [(300, 129, 77), (1000, 1002, 998), (520, 1004, 996)])
def test_pair_kernel_small_integers_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + N + K)
    C = rtm.gemm_bf16f32(A.to(torch.bfloat16).to(DEV), B.to(torch.bfloat16).to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


# C rows off 16-byte boundaries (N % 4 != 0) or fewer than 64 K-blocks: the
# TMA pair kernel behind the workspace entry point does not split K there.
@pytest.mark.parametrize("M,N,K", [(300, 129, 77), (1000, 1002, 998), (520, 1004, 996),
                                   (2000, 2002, 4998), (4097, 3001, 1023)])
def test_pair_kernel_bits_equal_repitched_tma_pair(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "bf16", seed=7 * M + N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    W = rtm.gemm_bf16f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.equal(C, W)


def test_pair_kernel_full_size_sampled():
    # 8192 x 8190 x 8190: rows on 4-byte boundaries (the workspace-free product
    # of that size).
    M, N, K = 8192, 8190, 8190
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=8190)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16", full=False, seed=3)
    again = rtm.gemm_bf16f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C, again)


def test_pair_kernel_f16_offset_operands():
    # fp16, A and B 2 bytes past a 16-byte boundary (2-byte accesses), C 4 bytes past.
    M, N, K = 600, 520, 264
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=52)
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

    pair_ran(call)
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert torch.isnan(Cb[0]) and torch.isnan(Cb[1 + M * N:]).all()
    assert_close_to_oracle(Cb[1:1 + M * N].view(M, N), A, B, "bf16")


def test_short_products_take_the_transposed_kernel():
    # M <= 128: C^T = B^T.A^T with the same producers, no CTA pair.
    M, N, K = 128, 1002, 998
    A, B = workloads.make_inputs(M, N, K, "normal", "bf16", seed=53)
    Ad, Bd = A.to(DEV), B.to(DEV)
    names = kernel_names(lambda: rtm.gemm_bf16f32(Ad, Bd))
    assert any("gemm_tc_any_t_kernel" in n for n in names), names
    assert not any(PAIR in n for n in names), names


@pytest.mark.parametrize("M,N,K", [(300, 258, 130), (520, 1004, 996), (257, 129, 77)],
                         ids=["pair_4byte", "pair_8byte_cp_async", "pair_2byte"])
def test_muted_producers_every_wait_gives_up(M, N, K):
    """The producer warps load nothing: every bounded wait (stage barriers, the
    odd CTA's forwarder, the accumulator barriers) runs out after 50 ms, the
    kernel records a timeout and returns, and the next product is correct."""
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
