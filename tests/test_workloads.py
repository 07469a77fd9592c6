"""CPU tests of the seeded input generators (no product arithmetic here)."""

import pytest
import torch

import workloads

pytestmark = pytest.mark.cpu


def test_inputs_are_seeded_and_shaped():
    A1, B1 = workloads.make_inputs(5, 7, 3, "uniform", "f32", seed=9)
    A2, B2 = workloads.make_inputs(5, 7, 3, "uniform", "f32", seed=9)
    assert A1.shape == (5, 3) and B1.shape == (3, 7)
    assert torch.equal(A1, A2) and torch.equal(B1, B2)
    assert A1.is_contiguous() and B1.is_contiguous()
    A3, _ = workloads.make_inputs(5, 7, 3, "uniform", "f32", seed=10)
    assert not torch.equal(A1, A3)


def test_distributions():
    A, B = workloads.make_inputs(256, 256, 256, "uniform", "f32", seed=1)
    assert A.dtype == torch.float32 and A.min() >= -1 and A.max() < 1
    A, _ = workloads.make_inputs(64, 64, 64, "int", "f32", seed=1)
    vals = set(A.flatten().tolist())
    assert vals <= set(float(v) for v in range(-4, 5)) and len(vals) == 9
    A, B = workloads.make_inputs(16, 16, 64, "normal", "bf16", seed=1)
    assert A.dtype == torch.bfloat16 and B.dtype == torch.bfloat16


def test_sample_indices_cover_edges():
    r, c = workloads.sample_indices(4097, 3001, count=4096, seed=2)
    assert r.dtype == torch.int64 and r.shape == c.shape
    assert int(r.min()) >= 0 and int(r.max()) < 4097 and int(c.max()) < 3001
    pairs = set(zip(r.tolist(), c.tolist()))
    for corner in [(0, 0), (0, 3000), (4096, 0), (4096, 3000)]:
        assert corner in pairs
    assert (r >= 4097 - 128).sum() >= 64 and (c >= 3001 - 128).sum() >= 64
    r0, c0 = workloads.sample_indices(0, 5)
    assert r0.numel() == 0 and c0.numel() == 0


def test_workload_table():
    w = workloads.WORKLOADS["bf16_8192_normal"]
    assert (w.M, w.N, w.K, w.dtype) == (8192, 8192, 8192, "bf16")
    assert w.flops == 2 * 8192 ** 3
    assert len({x.seed for x in workloads.WORKLOADS.values()}) == len(workloads.WORKLOADS)
