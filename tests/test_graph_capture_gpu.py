"""The product entry points can be captured into a CUDA graph once they have
run on the device (the per-device caches, including the cluster occupancy
queries of the split schedules, are then filled): a replay with new
inputs written into the captured buffers gives bit for bit what an eager call
gives, and agrees with the oracle."""

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_close_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


def _ws_f32(M, N, K):
    return torch.empty(max(rtm.gemm_f32_workspace_bytes(M, N, K) // 4, 1), device=DEV)


def _ws_2byte(M, N, K):
    return torch.empty(max(rtm.gemm_bf16f32_workspace_bytes(M, N, K), 1), dtype=torch.uint8,
                       device=DEV)


CASES = {
    # name: (dtype, M, N, K, call(A, B, C, workspace))
    "gemm_f32": ("f32", 640, 520, 384, lambda A, B, C, W: rtm.gemm_f32(A, B, out=C)),
    "gemm_f32 cluster split-K": ("f32", 1000, 1000, 999,
                                 lambda A, B, C, W: rtm.gemm_f32(A, B, out=C)),
    "gemm_f32 256x64 tiles, cluster split-K": ("f32", 8192, 64, 1024,
                                               lambda A, B, C, W: rtm.gemm_f32(A, B, out=C)),
    "gemm_f32_ws split-K": ("f32", 512, 64, 2048,
                            lambda A, B, C, W: rtm.gemm_f32_ws(A, B, out=C, workspace=W)),
    "gemm_f32_ws stream-K": ("f32", 1024, 1024, 1024,
                             lambda A, B, C, W: rtm.gemm_f32_ws(A, B, out=C, workspace=W)),
    "gemm_bf16f32 CTA pairs": ("bf16", 512, 512, 256,
                               lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
    "gemm_bf16f32 CTA pairs, K split": ("bf16", 256, 1024, 4096,
                                        lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
    "gemm_bf16f32 single CTA": ("bf16", 96, 2048, 512,
                                lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
    "gemm_bf16f32_ws re-pitched": ("bf16", 300, 129, 77,
                                   lambda A, B, C, W: rtm.gemm_bf16f32_ws(A, B, out=C,
                                                                          workspace=W)),
    "gemm_bf16f32 transposed, K split": ("bf16", 64, 4096, 4096,
                                         lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
    "gemm_f16f32 load-and-swizzle, transposed": ("f16", 100, 130, 90,
                                                 lambda A, B, C, W: rtm.gemm_f16f32(A, B, out=C)),
    "gemm_bf16f32 load-and-swizzle, transposed, K split": (
        "bf16", 16, 4094, 4094, lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
    "gemm_bf16f32 load-and-swizzle CTA pairs": ("bf16", 300, 258, 130,
                                                lambda A, B, C, W: rtm.gemm_bf16f32(A, B, out=C)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_capture_and_replay(name):
    dtype, M, N, K, call = CASES[name]
    A0, B0 = workloads.make_inputs(M, N, K, "normal", dtype, seed=M + N + K)
    A1, B1 = workloads.make_inputs(M, N, K, "normal", dtype, seed=M + N + K + 1)
    A, B = A0.to(DEV), B0.to(DEV)
    C = torch.empty(M, N, device=DEV)
    W = _ws_f32(M, N, K) if dtype == "f32" else _ws_2byte(M, N, K)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(A, B, C, W)  # fills the per-device caches outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(A, B, C, W)

    for A_host, B_host in ((A0, B0), (A1, B1)):
        A.copy_(A_host.to(DEV))
        B.copy_(B_host.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        replayed = C.clone()
        eager = torch.empty_like(C)
        call(A, B, eager, W)
        torch.cuda.synchronize()
        assert rtm.get_device_error() == 0
        assert torch.equal(replayed, eager), "replay differs from an eager call"
        assert_close_to_oracle(replayed, A_host, B_host, "bf16" if dtype != "f32" else "f32")
