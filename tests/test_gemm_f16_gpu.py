"""GPU parity tests of gemm_f16f32 (tcgen05 kernel, fp16 operands, fp32
accumulate) against the CPU oracle fed the same fp16 values."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_bit_exact, assert_close_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def run(A, B):
    C = rtm.gemm_f16f32(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    return C


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (1024, 1024, 1024), (1000, 1000, 1000),
                                   (129, 264, 72), (1, 8, 8), (2048, 4096, 512),
                                   (300, 129, 77), (1000, 999, 1001)])
def test_parity_shapes(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", "f16", seed=M + N + K)
    full = M * N * K <= (1 << 31)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=full, seed=M)


def test_full_size_sampled():
    A, B = workloads.make_inputs(8192, 8192, 8192, "normal", "f16", seed=workloads.SEED_BASE + 90)
    assert_close_to_oracle(run(A, B), A, B, "bf16", full=False, seed=90)


@pytest.mark.parametrize("M,N,K", [(200, 136, 1000), (257, 264, 8)])
def test_small_integer_bit_exact(M, N, K):
    A, B = workloads.make_inputs(M, N, K, "int", "f32", seed=M + K)
    C = run(A.to(torch.float16), B.to(torch.float16))
    assert_bit_exact(C, (A.to(torch.int64) @ B.to(torch.int64)).numpy())


def test_identity_exact():
    g = torch.Generator().manual_seed(91)
    A = torch.randn(384, 256, generator=g).to(torch.float16)
    assert_bit_exact(run(A, torch.eye(256).to(torch.float16)), A.float().numpy())


def test_fp16_differs_from_bf16_path():
    """Same bit patterns read as fp16 and as bf16 give different products:
    the format field reaches the tensor core."""
    A, B = workloads.make_inputs(128, 256, 64, "int", "f32", seed=92)
    Ah, Bh = A.to(torch.float16).to(DEV), B.to(torch.float16).to(DEV)
    Ch = rtm.gemm_f16f32(Ah, Bh)
    Cb = rtm.gemm_bf16f32(Ah.view(torch.bfloat16), Bh.view(torch.bfloat16))
    torch.cuda.synchronize()
    assert not torch.equal(Ch, Cb)
