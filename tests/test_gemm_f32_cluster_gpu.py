"""GPU tests of the fp32 split-K over thread-block clusters: products with too
few C tiles to fill the GPU, run through gemm_f32 (no workspace), split K over
2, 4 or 8 CTAs of one cluster, which add their partial tiles through
distributed shared memory in rank order. Each shape below was chosen so the
schedule on a 152-SM GB300 takes the variant named beside it (cluster size,
one CTA per SM or two, tile shape, 16-byte or 4-byte paths); every one is
checked against the oracle."""

import numpy as np
import pytest
import torch

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


SHAPES = [
    (300, 3000, 700),    # 2 per cluster
    (300, 700, 400),     # 64 x 64 tiles (the plan's choice for few tiles), 2 per cluster
    (1024, 1024, 1024),  # 4 per cluster, two CTAs per SM
    (1000, 1000, 999),   # the same, ragged in M, N and K
    (512, 512, 512),     # 4 per cluster, one CTA per SM
    (640, 520, 384),     # 4 per cluster, ragged N, three slices per chunk
    (256, 256, 256),     # 8 per cluster spread one CTA per SM, one slice per chunk
    (300, 200, 1024),    # 8 per cluster spread, ragged tiles
    (129, 65, 999),      # 8 per cluster spread, one spare row and column tile
    (4096, 64, 4096),    # 128 x 64 tiles, 8 per cluster, two CTAs per SM
    (48, 4096, 4096),    # 64 x 128 tiles, 8 per cluster, two CTAs per SM
    (64, 8, 4096),       # 64 x 64 tiles, 8 per cluster spread
    (48, 64, 1000),      # 64 x 64 tiles, 8 per cluster spread, partial last chunk
    (300, 201, 1024),    # N % 4 != 0: 4-byte copies of B and stores of C
    (1200, 1300, 700),   # 4 per cluster, three waves of CTAs
    (2048, 640, 2048),   # 8 per cluster, five waves of CTAs
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_cluster_split_parity(M, N, K):
    kind, splits = rtm.gemm_f32_schedule(M, N, K)
    assert kind == "tiles+cluster-split" and splits in (2, 4, 8), (kind, splits)
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 31 + N * 7 + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


# Tall, narrow products (N <= 64) on 256 x 64 tiles, 16 x 4 outputs per
# thread, K split over a cluster or not at all.
TALL_SHAPES = [
    (8192, 64, 4096, 8),    # 32 tiles, 8 per cluster, two CTAs per SM
    (8193, 64, 2048, 8),    # one spare row: a 256-row tile with a single live row
    (16384, 64, 2048, 4),   # 64 tiles, 4 per cluster
    (8192, 61, 4096, 8),    # rows of B off 16-byte boundaries: 128 x 64 tiles, same split
    (3000, 33, 1500, 8),    # 12 tiles spread one CTA per SM, ragged in M, N and K
    (32768, 64, 512, 1),    # 128 tiles unsplit
    (20000, 64, 300, 1),    # more tiles than SMs, ragged M and K
]


@pytest.mark.parametrize("M,N,K,splits", TALL_SHAPES)
def test_tall_tiles_parity(M, N, K, splits):
    kind, s = rtm.gemm_f32_schedule(M, N, K)
    want = "tall-tiles+cluster-split" if splits > 1 else "tall-tiles"
    assert (kind, s) == (want, splits), (kind, s)
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 13 + N * 5 + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


# Products of 33 to 64 rows on 64 x 256 tiles, 4 x 16 outputs per thread.
WIDE_SHAPES = [
    (64, 8192, 4096, 8),    # 32 tiles, 8 per cluster, two CTAs per SM
    (60, 3000, 2000, 8),    # 12 tiles, 8 per cluster spread, ragged M, N and K
    (60, 8192, 2048, 8),    # a 60-row tile
    (64, 16384, 2048, 4),   # 64 tiles, 4 per cluster
    (40, 8192, 4096, 8),    # 40 live rows of 64
    (64, 8191, 4096, 8),    # N % 4 != 0: 4-byte copies of B and stores of C
    (64, 65536, 512, 1),    # 256 tiles unsplit
]


@pytest.mark.parametrize("M,N,K,splits", WIDE_SHAPES)
def test_wide_tiles_parity(M, N, K, splits):
    kind, s = rtm.gemm_f32_schedule(M, N, K)
    want = "wide-tiles+cluster-split" if splits > 1 else "wide-tiles"
    assert (kind, s) == (want, splits), (kind, s)
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 11 + N * 3 + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


def test_wide_tiles_sampled_64x8192x8192():
    M, N, K = 64, 8192, 8192
    assert rtm.gemm_f32_schedule(M, N, K) == ("wide-tiles+cluster-split", 8)
    assert rtm.gemm_f32_workspace_bytes(M, N, K) == 0  # the workspace split prices higher
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=85)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = rtm.gemm_f32(Ad, Bd)
    Cw = rtm.gemm_f32_ws(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C, Cw)
    assert_close_to_oracle(C, A, B, "f32", full=False, seed=85)


@pytest.mark.parametrize("M,N,K", [(60, 3000, 2000), (64, 8192, 1024), (64, 65536, 512)])
def test_wide_tiles_small_integer_guard_band_repeatability(M, N, K):
    A, B = small_int_inputs(M, N, K, seed=M + 5 * K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32(Ad, Bd, out=C)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N), "a store landed outside C"
    assert torch.equal(C, C2)
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


@pytest.mark.parametrize("M,N,K", [(8193, 64, 2048), (8192, 64, 1024), (20000, 64, 300)])
def test_tall_tiles_small_integer_guard_band_repeatability(M, N, K):
    A, B = small_int_inputs(M, N, K, seed=M + 7 * K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32(Ad, Bd, out=C)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N), "a store landed outside C"
    assert torch.equal(C, C2)
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_tall_tiles_unaligned_output():
    # C starts 4 bytes past a 16-byte boundary: 4-byte stores on the 256-row tiles.
    M, N, K = 8192, 64, 1024
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=6)
    buf = torch.full((M * N + 4,), float("nan"), device=DEV)
    C = buf[1:1 + M * N].view(M, N)
    rtm.gemm_f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + M * N:]).all()
    assert_close_to_oracle(C, A, B, "f32")


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1000, 1000, 999), (48, 64, 1000),
                                   (2048, 640, 2048)])
def test_cluster_split_small_integer_bit_exact(M, N, K):
    A, B = small_int_inputs(M, N, K, seed=M + N + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


@pytest.mark.parametrize("M,N,K", [(300, 200, 1024), (129, 65, 999), (1000, 1000, 999)])
def test_cluster_split_guard_band_and_repeatability(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32(Ad, Bd, out=C)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N), "a store landed outside C"
    assert torch.equal(C, C2), "the rank-ordered sum repeats exactly"
    assert_close_to_oracle(C, A, B, "f32")


def test_cluster_split_unaligned_output():
    # C starts 4 bytes past a 16-byte boundary: the 4-byte store path.
    M, N, K = 640, 520, 384
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=5)
    buf = torch.full((M * N + 4,), float("nan"), device=DEV)
    C = buf[1:1 + M * N].view(M, N)
    rtm.gemm_f32(A.to(DEV), B.to(DEV), out=C)
    torch.cuda.synchronize()
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + M * N:]).all()
    assert_close_to_oracle(C, A, B, "f32")


def test_workspace_entry_takes_the_cheaper_split():
    # gemm_f32 splits 1024^3 and 512 x 512 x 8192 over clusters (no
    # workspace); gemm_f32_ws runs them as stream-K through its workspace.
    # 1000 x 1000 x 999 takes the cluster split through both (gemm_f32_ws on a
    # copy of A re-pitched into its workspace, the only workspace it uses, for
    # the TMA-fed kernels: the same sums), and 256 x 256 x 2048 the workspace
    # split.
    assert rtm.gemm_f32_schedule(1024, 1024, 1024)[0] == "tiles+cluster-split"
    assert rtm.gemm_f32_schedule(1024, 1024, 1024, workspace=True)[0] == "tiles+stream-k"
    assert rtm.gemm_f32_workspace_bytes(512, 512, 8192) > 0
    assert rtm.gemm_f32_schedule(512, 512, 8192, workspace=True)[0] == "tiles+stream-k"
    assert rtm.gemm_f32_schedule(512, 512, 8192)[0] == "tiles+cluster-split"
    assert rtm.gemm_f32_workspace_bytes(1000, 1000, 999) == (1000 * 1000 * 4 + 255) // 256 * 256
    assert rtm.gemm_f32_schedule(1000, 1000, 999, workspace=True)[0] == "tiles+cluster-split"
    assert rtm.gemm_f32_schedule(256, 256, 2048, workspace=True)[0] == "tiles+workspace-split"
    assert rtm.gemm_f32_schedule(16, 8192, 8192)[0] == "column-strips"
    for M, N, K in [(1024, 1024, 1024), (512, 512, 8192), (1000, 1000, 999), (256, 256, 2048)]:
        A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + K)
        Ad, Bd = A.to(DEV), B.to(DEV)
        Cw = rtm.gemm_f32_ws(Ad, Bd)
        C = rtm.gemm_f32(Ad, Bd)
        torch.cuda.synchronize()
        assert_close_to_oracle(Cw, A, B, "f32")
        assert_close_to_oracle(C, A, B, "f32")
        if K == 999:
            assert torch.equal(C, Cw), "both entries run the same schedule"


# More tiles than SMs: whole waves of tiles unsplit, then the ragged last wave
# with K split over clusters of 4 (a second launch starting at a tile offset).
TAIL_SHAPES = [
    (2048, 1536, 1024),  # 192 tiles, fewer than two waves: all of them split
    (3072, 2048, 1000),  # 304 tiles unsplit + 80 split, ragged K
    (2050, 1540, 1100),  # 221 edge-heavy tiles, 9-slice chunks, ragged K
]


@pytest.mark.parametrize("M,N,K", TAIL_SHAPES)
def test_tail_split_parity(M, N, K):
    kind, splits = rtm.gemm_f32_schedule(M, N, K)
    assert kind == "tiles+tail-cluster-split" and splits == 4, (kind, splits)
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + 3 * N + K)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


def test_tail_split_config_4097x3001x1023_sampled():
    """The ragged 4097 x 3001 x 1023 workload: 608 tiles unsplit, 184 split."""
    w = workloads.WORKLOADS["f32_4097x3001x1023"]
    assert rtm.gemm_f32_schedule(w.M, w.N, w.K)[0] == "tiles+tail-cluster-split"
    A, B = workloads.workload_inputs(w)
    C = rtm.gemm_f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert_close_to_oracle(C, A, B, "f32", full=False, seed=w.seed)


def test_tail_split_small_integer_guard_band_repeatability():
    M, N, K = 2050, 1540, 1100
    A, B = small_int_inputs(M, N, K, seed=52)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    rtm.gemm_f32(Ad, Bd, out=C)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert guard_intact(buf, M, N)
    assert torch.equal(C, C2)
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_tail_split_rule_leaves_these_unsplit():
    assert rtm.gemm_f32_schedule(4096, 4096, 4096) == ("tiles", 1)  # 112-tile tail after 3 waves
    assert rtm.gemm_f32_schedule(8192, 8192, 8192) == ("tiles", 1)
    assert rtm.gemm_f32_schedule(2048, 2304, 512) == ("tiles", 1)   # 4-slice chunks, 95 % full
