"""GPU tests of the TMA-fed rectangular-tile fp32 kernel (simt_tma_rect):
256 x 64 C tiles (16 x 4 outputs per thread) for tall, narrow products and
64 x 256 tiles (4 x 16) for products of 33-64 rows, K split over a cluster or
unsplit, which gemm_f32 runs where the TMA unit can address the rows (K % 4
== 0, N % 4 == 0, A and B 16-byte aligned).

Checked: the kernel that runs, the oracle (|C - C_oracle| <= 1e-4 * sum_k
|A[i][k] B[k][j]|), a NaN guard band around C, and bit equality with the
cp.async-fed kernel, which gemm_f32 runs when B starts 4 bytes past a
16-byte boundary: same split, same K order per element, and the packed FMA
rounds each half like a scalar fmaf."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_close_to_oracle, guard_intact, guarded_output, kernel_names

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (M, N, K, splits, schedule): ragged rows (a tile with one live row), ragged
# K (300 = 9 slices + 12), narrower tiles (48 of 64 columns, 40 or 60 of 64
# rows), splits 1 to 8.
SHAPES = [(8192, 64, 4096, 8, "tall"), (8193, 64, 2048, 8, "tall"), (16384, 64, 2048, 4, "tall"),
          (32768, 64, 512, 1, "tall"), (20000, 64, 300, 1, "tall"), (8192, 48, 4096, 8, "tall"),
          (64, 8192, 4096, 8, "wide"), (60, 3000, 2000, 8, "wide"), (40, 8192, 4096, 8, "wide"),
          (64, 16384, 2048, 4, "wide"), (64, 65536, 512, 1, "wide")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def offset_copy(B):
    """B on the device, 4 bytes past a 16-byte boundary."""
    K, N = B.shape
    buf = torch.empty(K * N + 1, device=DEV)
    Bo = buf[1:].view(K, N)
    Bo.copy_(B.to(DEV))
    return Bo


@pytest.mark.parametrize("M,N,K,splits,shape", SHAPES)
def test_rect_tma_kernel_matches_oracle_and_cp_async_bits(M, N, K, splits, shape):
    kind, s = rtm.gemm_f32_schedule(M, N, K)
    assert s == splits and kind.startswith(shape + "-tiles"), (kind, s)
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M + 3 * N + K)
    Ad, Bd = A.to(DEV), B.to(DEV)
    buf, C = guarded_output(M, N, DEV)
    names = kernel_names(lambda: rtm.gemm_f32(Ad, Bd, out=C))
    assert any("simt_tma_rect::" in n for n in names), names
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert guard_intact(buf, M, N)
    assert_close_to_oracle(C, A, B, "f32", full=M * N * K <= (1 << 31), seed=M)
    Bo = offset_copy(B)
    names = kernel_names(lambda: rtm.gemm_f32(Ad, Bo))
    assert not any("simt_tma_rect::" in n for n in names), names
    C_ref = rtm.gemm_f32(Ad, Bo)
    torch.cuda.synchronize()
    assert torch.equal(C, C_ref), "TMA-fed and cp.async-fed tiles must agree bit for bit"


@pytest.mark.parametrize("M,N,K", [(8192, 64, 4096), (64, 8192, 4096)])
def test_rect_tma_kernel_repeats_bit_for_bit(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "f32", seed=91)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = rtm.gemm_f32(Ad, Bd)
    C2 = rtm.gemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
