"""Seeded shape fuzz: every entry point on many random shapes against the full
CPU oracle. Shapes mix tiny, ragged and tile-multiple sizes; for the tensor-
core entry points they cover both the TMA path (K, N multiples of 8) and the
load-and-swizzle or re-pitched path (anything else)."""

import random

import pytest
import torch

import register_tiled_matrix_gb300 as rtm
import workloads
from tests.parity import assert_close_to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _shapes(seed, count, lo=1, hi=700):
    rng = random.Random(seed)
    pool = [1, 2, 7, 8, 15, 16, 31, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 513]
    out = []
    for _ in range(count):
        dims = []
        for _ in range(3):
            dims.append(rng.choice(pool) if rng.random() < 0.5 else rng.randint(lo, hi))
        out.append(tuple(dims))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rtm.build()
    rtm.load_library()


F32_ENTRIES = {
    "gemm_f32": lambda A, B: rtm.gemm_f32(A, B),
    "gemm_f32_ws": lambda A, B: rtm.gemm_f32_ws(A, B),
    "ladder_2": lambda A, B: rtm.gemm_f32_ladder(2, A, B),
}


@pytest.mark.parametrize("entry", list(F32_ENTRIES))
@pytest.mark.parametrize("M,N,K", _shapes(2024, 16))
def test_fuzz_f32(entry, M, N, K):
    A, B = workloads.make_inputs(M, N, K, "uniform", "f32", seed=M * 1000003 + N * 1009 + K)
    C = F32_ENTRIES[entry](A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "f32")


def _tc_shapes(seed, count):
    rng = random.Random(seed)
    out = []
    for i in range(count):
        M = rng.randint(1, 600)
        if i % 2 == 0:   # TMA path: K, N multiples of 8
            N, K = 8 * rng.randint(1, 80), 8 * rng.randint(1, 80)
        else:            # load-and-swizzle path
            N, K = rng.randint(1, 600), rng.randint(1, 600)
        out.append((M, N, K))
    return out


TC_ENTRIES = {
    "gemm_bf16f32": ("bf16", rtm.gemm_bf16f32),
    "gemm_f16f32": ("f16", rtm.gemm_f16f32),
    "gemm_bf16f32_ws": ("bf16", rtm.gemm_bf16f32_ws),
    "gemm_f16f32_ws": ("f16", rtm.gemm_f16f32_ws),
}


@pytest.mark.parametrize("entry", list(TC_ENTRIES))
@pytest.mark.parametrize("M,N,K", _tc_shapes(2025, 14))
def test_fuzz_tensor_core(entry, M, N, K):
    dtype, fn = TC_ENTRIES[entry]
    A, B = workloads.make_inputs(M, N, K, "normal", dtype, seed=M * 7919 + N * 31 + K)
    C = fn(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")


def _long_k_shapes(seed, count):
    """Long K (2048..3072, a multiple of 8) with one short side: the kernel that
    splits K over a cluster, in both orientations."""
    rng = random.Random(seed)
    out = []
    for i in range(count):
        K = 8 * rng.randint(256, 384)
        if i % 2 == 0:   # short, wide
            M, N = rng.randint(1, 128), 8 * rng.randint(1, 256)
        else:            # tall, narrow
            M, N = rng.randint(129, 1500), 8 * rng.randint(1, 32)
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", _long_k_shapes(2026, 8))
def test_fuzz_long_k_one_short_side(dtype, M, N, K):
    A, B = workloads.make_inputs(M, N, K, "normal", dtype, seed=M * 131 + N * 7 + K)
    fn = rtm.gemm_bf16f32 if dtype == "bf16" else rtm.gemm_f16f32
    C = fn(A.to(DEV), B.to(DEV))
    torch.cuda.synchronize()
    assert rtm.get_device_error() == 0
    assert_close_to_oracle(C, A, B, "bf16")
