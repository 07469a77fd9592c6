"""CPU tests: the oracle against its pins, and mutated oracles against the pins.

The oracle computes the plain definition of the product
(C[i][j] = sum_k A[i][k] B[k][j]; "【infra之路】理解 Register Tiling", section
"先看 Shared Memory 版本里，一个线程在做什么"). Before it is trusted it is pinned
to exact rational arithmetic, integer products and closed forms
(tests/oracle_pins.py). To show that the pins would catch a plausible slip,
copies of oracle.c with a planted mistake are compiled here on the CPU and
each must fail at least one pin.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from tests import oracle_pins

pytestmark = pytest.mark.cpu


def _gemm(A, B):
    return oracle.gemm(A, B)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_meets_pin(pin):
    pin(_gemm)


def test_sampled_matches_full():
    A, B = workloads.make_inputs(37, 29, 41, "uniform", "f32", seed=3)
    C, S = oracle.gemm(A, B)
    rows, cols = workloads.sample_indices(37, 29, count=200, seed=3, edge=8, edge_count=10)
    Cs, Ss = oracle.gemm_sampled(A, B, rows, cols)
    assert np.array_equal(Cs, C[rows.numpy(), cols.numpy()])
    assert np.array_equal(Ss, S[rows.numpy(), cols.numpy()])


def test_thread_count_does_not_change_result():
    A, B = workloads.make_inputs(64, 48, 300, "normal", "f32", seed=4)
    C1, S1 = oracle.gemm(A, B, threads=1)
    C4, S4 = oracle.gemm(A, B, threads=4)
    assert np.array_equal(C1, C4) and np.array_equal(S1, S4)
    assert oracle.max_threads() >= 1


def test_bf16_inputs_widen_exactly():
    A, B = workloads.make_inputs(8, 8, 16, "normal", "bf16", seed=5)
    C, _ = oracle.gemm(A, B)
    C2, _ = oracle.gemm(A.float(), B.float())
    assert np.array_equal(C, C2)


def test_sampled_rejects_out_of_range():
    A, B = workloads.make_inputs(4, 4, 4, "uniform", "f32", seed=6)
    with pytest.raises(IndexError):
        oracle.gemm_sampled(A, B, [4], [0])


# --- planted mistakes ------------------------------------------------------
# (name, text in oracle.c, replacement). Each must make some pin fail.
MUTANTS = [
    ("transposed_B", "(double)B[k * N + j]", "(double)B[(j * K + k) % (K * N)]"),
    ("dropped_last_term", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)"),
    ("dropped_first_term", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    ("sign_flip", "c += p;", "c -= p;"),
    ("A_index_shift", "(double)A[i * K + k]", "(double)A[i * K + (k + 1) % K]"),
    ("S_without_abs", "s += fabs(p);", "s += p;"),
    ("fp32_accumulator", "double c = 0.0;", "float c = 0.0f;"),
    ("row_col_swap", "&C[i * N + j], &S[i * N + j]", "&C[(j * M + i) % (M * N)], &S[i * N + j]"),
]


@pytest.fixture(scope="module")
def oracle_source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, oracle_source, name, old, new):
    assert old in oracle_source, f"mutation site for {name} not found"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(oracle_source.replace(old, new))
    so = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(src), "-o", str(so), "-lm"], check=True)
    lib = oracle.bind(ctypes.CDLL(str(so)))
    failed = oracle_pins.failing_pins(lambda A, B: oracle.gemm(A, B, lib=lib))
    assert failed, f"mutant {name} passed every pin"
