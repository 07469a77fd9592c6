"""GPU parity tests of gemm_f32 (SIMT FP32 register-tiled kernel) against the
CPU oracle, through the C ABI (ctypes binding)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import (assert_bit_exact, assert_close_to_oracle, guard_intact,
                          guarded_output, small_int_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def run(A, B):
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    return C


F32_WORKLOADS = [w for w in workloads.WORKLOADS.values() if w.dtype == "f32" and w.dist != "int"]


@pytest.mark.parametrize("w", F32_WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(w):
    A, B = workloads.workload_inputs(w)
    C = run(A, B)
    assert_close_to_oracle(C, A, B, "f32", full=w.full_check, seed=w.seed)


def test_small_integer_workload_bit_exact():
    w = workloads.WORKLOADS["f32_256_int"]
    A, B = workloads.workload_inputs(w)
    C = run(A, B)
    C0, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C0)


SHAPES = [(1, 1, 1), (1, 257, 1), (129, 1, 17), (7, 5, 3), (128, 128, 16), (127, 129, 15),
          (129, 127, 17), (131, 257, 33), (256, 384, 100), (37, 4, 1000), (300, 301, 302),
          (65, 1000, 31)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_integer_bit_exact_ragged(M, N, K):
    A, B = small_int_inputs(M, N, K, seed=M * 7 + N * 3 + K)
    C = run(A, B)
    expect = (A.to(torch.int64) @ B.to(torch.int64)).numpy()
    assert_bit_exact(C, expect)


@pytest.mark.parametrize("M,N,K", [(300, 200, 129), (513, 260, 64), (64, 64, 4096)])
def test_uniform_ragged_parity(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + N + K)
    assert_close_to_oracle(run(A, B), A, B, "f32")


def test_identity_and_permutation_exact():
    g = torch.Generator().manual_seed(21)
    A = torch.randn(300, 200, generator=g)
    I = torch.eye(200)
    assert_bit_exact(run(A, I), A.numpy())
    assert_bit_exact(run(torch.eye(300), A), A.numpy())
    p = torch.randperm(300, generator=g)
    P = torch.zeros(300, 300)
    P[torch.arange(300), p] = 1.0
    assert_bit_exact(run(P, A), A[p].numpy())
    q = torch.randperm(200, generator=g)
    Q = torch.zeros(200, 200)
    Q[q, torch.arange(200)] = 1.0
    assert_bit_exact(run(A, Q), A[:, q].numpy())


def test_rank_one_closed_form():
    g = torch.Generator().manual_seed(22)
    M, N, K = 200, 150, 513
    u = torch.randint(-30, 31, (M,), generator=g).float()
    v = torch.randint(-30, 31, (N,), generator=g).float()
    A = u[:, None].expand(M, K).contiguous()
    B = v[None, :].expand(K, N).contiguous()
    assert_bit_exact(run(A, B), (K * torch.outer(u, v)).numpy())


def test_transpose_and_linearity():
    A, B = workloads.make_inputs(257, 190, 300, "uniform", "f32", seed=23)
    C = run(A, B).cpu()
    Ct = run(B.t().contiguous(), A.t().contiguous()).cpu()
    _, S = oracle.gemm(A, B)
    S = torch.from_numpy(S).float()
    assert torch.all((C - Ct.t()).abs() <= 2e-4 * S)
    B2 = workloads.make_inputs(257, 190, 300, "uniform", "f32", seed=24)[1]
    lhs = run(A, B + B2).cpu()
    rhs = C + run(A, B2).cpu()
    _, S2 = oracle.gemm(A, (B.abs() + B2.abs()))
    assert torch.all((lhs - rhs).abs() <= 3e-4 * torch.from_numpy(S2).float())


def test_k_zero_writes_zeros_and_empty_is_noop():
    C = torch.full((5, 7), 3.0, device=DEV)
    rtm.gemm_f32(torch.empty(5, 0, device=DEV), torch.empty(0, 7, device=DEV), out=C)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0
    lib = rtm.load_library()
    buf = torch.full((16,), 5.0, device=DEV)
    assert lib.gemm_f32(0, 4, 4, None, None, buf.data_ptr(), None) == 0
    assert lib.gemm_f32(4, 0, 4, None, None, buf.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert torch.all(buf == 5.0)


@pytest.mark.parametrize("M,N,K", [(200, 257, 99), (128, 128, 128), (1, 3001, 7)])
def test_guard_band_untouched(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=31)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "f32")


def test_unaligned_pointers_take_scalar_paths():
    """Operands at a 4-byte (not 16-byte) offset: B and C use the 4-byte paths."""
    M, N, K = 190, 132, 77
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=32)
    Ab = torch.zeros(M * K + 1, device=DEV)
    Bb = torch.zeros(K * N + 1, device=DEV)
    Cb = torch.zeros(M * N + 1, device=DEV)
    Ab[1:] = A.flatten().to(DEV)
    Bb[1:] = B.flatten().to(DEV)
    lib = rtm.load_library()
    st = lib.gemm_f32(M, N, K, Ab.data_ptr() + 4, Bb.data_ptr() + 4, Cb.data_ptr() + 4,
                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert_close_to_oracle(Cb[1:].view(M, N), A, B, "f32")


def test_repeated_calls_identical():
    A, B = workloads.make_inputs(1024, 512, 768, "normal", "f32", seed=33)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = rtm.gemm_f32(Ad, Bd)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2), "the kernel is deterministic: same inputs, same bits"


def test_on_side_stream():
    A, B = workloads.make_inputs(512, 512, 512, "uniform", "f32", seed=34)
    s = torch.cuda.Stream()
    Ad, Bd = A.to(DEV), B.to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = rtm.gemm_f32(Ad, Bd)
    s.synchronize()
    assert_close_to_oracle(C, A, B, "f32")


@pytest.mark.parametrize("N", [1, 17, 33, 63, 64, 65])
def test_narrow_tile_boundary(N):
    """N <= 64 runs 128 x 64 tiles, N > 64 128 x 128 tiles; exercise both sides."""
    M, K = 300, 257
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=N)
    assert_close_to_oracle(run(A, B), A, B, "f32")
    Ai, Bi = small_int_inputs(M, N, K, seed=N + 1)
    assert_bit_exact(run(Ai, Bi), (Ai.to(torch.int64) @ Bi.to(torch.int64)).numpy())


# M <= 32: two columns of C per thread, K split over S CTAs of a cluster
# (S for a 152-SM GPU noted: up to two CTAs per SM, S = 8 when every cluster
# of 8 is resident); no workspace in any fp32 entry point.
@pytest.mark.parametrize("M,N,K", [(1, 8192, 4096),    # S = 8: clusters of 8
                                   (7, 1000, 999),     # S = 2
                                   (16, 257, 3000),    # S = 8, 4-byte B copies
                                   (32, 4096, 8192),   # S = 8
                                   (17, 64, 33),       # 32 accumulators, one CTA
                                   (1, 1, 1),
                                   (9, 8190, 2048),    # S = 8, 4-byte B copies
                                   (32, 2048, 8192),   # S = 8
                                   (8, 16384, 4096),   # S = 4
                                   (9, 12290, 2048)])  # S = 4, 4-byte B copies
def test_short_wide_parity(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 31 + N + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "f32")


def test_short_wide_small_integer_bit_exact():
    A, B = small_int_inputs(24, 1000, 4096, seed=81)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_short_wide_guard_band_repeatability_and_entry_points():
    M, N, K = 20, 300, 2000
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=82)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV, pad=4096)
    rtm.gemm_f32(Ad, Bd, out=C)
    C2 = rtm.gemm_f32(Ad, Bd)
    assert rtm.gemm_f32_workspace_bytes(M, N, K) == 0
    C3 = rtm.gemm_f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert torch.equal(C, C2) and torch.equal(C, C3)
    assert_close_to_oracle(C, A, B, "f32")


# 32 < M <= 64: 64-row tiles (64 x 128 or 64 x 256, or 64 x 64 for N <= 64),
# plain and with K split over a workspace.
@pytest.mark.parametrize("M,N,K", [(33, 8192, 4096), (64, 1000, 999), (48, 64, 1000),
                                   (40, 130, 77), (64, 257, 2048)])
def test_64_row_tiles_parity(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 17 + N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_f32(Ad, Bd)
    Cw = rtm.gemm_f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "f32")
    assert_close_to_oracle(Cw, A, B, "f32")


def test_64_row_tiles_sampled_and_bit_exact():
    M, N, K = 64, 4096, 8192
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=83)
    assert rtm.gemm_f32_workspace_bytes(M, N, K) > 0
    C = rtm.gemm_f32_ws(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "f32", full=False, seed=83)
    Ai, Bi = small_int_inputs(50, 300, 4096, seed=84)
    Ci = rtm.gemm_f32_ws(Ai.to(DEV), Bi.to(DEV))
    torch.cuda.synchronize()
    assert_bit_exact(Ci, (Ai.to(torch.int64) @ Bi.to(torch.int64)).numpy())
