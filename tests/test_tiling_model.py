"""CPU tests of the counting model of the register-tiling page's kernels.

The model (oracle/tiling_model.py) runs the page's loops with read counters.
Its product must equal the plain oracle's (tiling re-groups the sum over k),
and its counters must reproduce the numbers the page prints
(tests/golden/register_tiling_counts.json, each entry cited)."""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import tiling_model as tm

pytestmark = pytest.mark.cpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "register_tiling_counts.json")))
G = {item["id"]: item for item in GOLDEN["items"]}


def _ints(M, N, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(-4, 5, (M, K)).astype(np.float32),
            rng.integers(-4, 5, (K, N)).astype(np.float32))


@pytest.fixture(scope="module")
def square64():
    A, B = _ints(64, 64, 64, 1)
    C0, _ = oracle.gemm(A, B)
    return A, B, C0


def test_naive_model(square64):
    A, B, C0 = square64
    C, c = tm.naive(A, B)
    assert np.array_equal(C, C0)
    N = 64
    assert c.per_output(64, 64)["global"] == 2 * N == eval(G["naive_global_reads_per_output"]["value_expr"])
    assert c.shared_reads == 0


def test_shared_tiled_model(square64):
    A, B, C0 = square64
    C, c = tm.shared_tiled(A, B, tile=32)
    assert np.array_equal(C, C0)
    N, TILE = 64, 32
    per = c.per_output(64, 64)
    tiles = N // TILE
    assert per["shared"] / tiles == G["shared_reads_per_output_per_tile"]["value"] == 64
    assert per["shared"] / tiles == eval(G["shared_shared_reads_per_output"]["value_expr"])
    assert per["shared"] / N == 2.0
    assert per["global"] == eval(G["shared_global_reads_per_output"]["value_expr"]) == N / 16


def test_register_tiled_model(square64):
    A, B, C0 = square64
    C, c = tm.register_tiled(A, B, threads=16, TM=4, TN=4, BK=16)
    assert np.array_equal(C, C0)
    per = c.per_output(64, 64)
    K = 64
    assert per["shared"] / K == G["register_shared_reads_per_output_per_k"]["value"] == 0.5
    assert per["fmas"] == K
    threads = 16 * 16
    assert threads == G["register_threads_per_block"]["value"]
    assert 16 * 4 == G["register_block_tile"]["value"]
    assert threads * 16 == G["register_outputs_per_block"]["value"]
    # per thread per k: TM + TN shared reads, TM * TN multiply-adds
    per_thread_per_k_reads = c.shared_reads / (threads * K)
    per_thread_per_k_fmas = c.fmas / (threads * K)
    assert per_thread_per_k_reads == G["register_shared_reads_per_thread_per_k"]["value"]
    assert per_thread_per_k_fmas == G["register_fmas_per_thread_per_k"]["value"]
    assert 4 * 4 + 4 + 4 == G["register_thread_registers"]["value"]
    assert 2.0 / (per["shared"] / K) == G["shared_vs_register_reduction"]["value"]
    # fewer global reads than the shared kernel ("每元素读 Global: 更少")
    assert per["global"] == tm.predicted_global_reads_per_output(K, 64, 64) < K / 16


def test_models_on_ragged_shape_match_oracle():
    A, B = _ints(37, 70, 45, 2)
    C0, _ = oracle.gemm(A, B)
    for fn in (tm.naive, lambda a, b: tm.shared_tiled(a, b, 32),
               lambda a, b: tm.register_tiled(a, b, 16, 4, 4, 16)):
        C, c = fn(A, B)
        assert np.array_equal(C, C0)
        assert c.fmas >= 37 * 70 * 45


def test_predictions_for_this_builds_tiles():
    assert tm.predicted_shared_reads_per_output_per_k(4, 4) == 0.5
    assert tm.predicted_shared_reads_per_output_per_k(8, 8) == 0.25
    assert tm.predicted_global_reads_per_output(4096, 128, 128) == 64.0
