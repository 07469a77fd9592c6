"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each pin takes `gemm(A, B) -> (C, S)` (fp64 numpy arrays) and raises
AssertionError when the callable disagrees with what mathematics fixes:

  exact_bound      brute force with exact rationals (fractions.Fraction) on
                   every shape 1 <= M, N, K <= 5: every fp32 value is a dyadic
                   rational, so the true sum is exact; a sequential fp64 sum
                   of exact fp64 products is within (K-1)*2^-53*S of it.
  identity         A.I == A and I.B == B bit for bit.
  permutation      P.A is A with rows permuted, A.P is A with columns
                   permuted, bit for bit.
  small_integer    entries in {-4..4}: C equals the int64 product and S the
                   int64 product of |A| and |B| (every partial sum < 2^53).
  rank_one         A = u.1^T, B = 1.v^T gives C[i][j] = K*u[i]*v[j].
  empty            K = 0 gives C = S = 0; M = 0 or N = 0 gives empty results.

None of them re-types the oracle's loop: the references are exact rational
arithmetic, integer matrix products and closed forms.
"""

from __future__ import annotations

import itertools
from fractions import Fraction
from typing import Callable, Tuple

import numpy as np

GemmFn = Callable[[np.ndarray, np.ndarray], Tuple[np.ndarray, np.ndarray]]


def _rand_f32(rng: np.random.Generator, shape) -> np.ndarray:
    # Mixed magnitudes and full 24-bit mantissas so fp64 sums really round.
    mant = rng.uniform(-1.0, 1.0, size=shape)
    expo = rng.integers(-6, 7, size=shape)
    return (mant * np.exp2(expo)).astype(np.float32)


def pin_exact_bound(gemm: GemmFn, max_dim: int = 5, seed: int = 11) -> None:
    rng = np.random.default_rng(seed)
    for M, N, K in itertools.product(range(1, max_dim + 1), repeat=3):
        A = _rand_f32(rng, (M, K))
        B = _rand_f32(rng, (K, N))
        C, S = gemm(A, B)
        assert C.shape == (M, N) and S.shape == (M, N), (M, N, K)
        Af = [[Fraction(float(v)) for v in row] for row in A]
        Bf = [[Fraction(float(v)) for v in row] for row in B]
        for i in range(M):
            for j in range(N):
                prods = [Af[i][k] * Bf[k][j] for k in range(K)]
                exact = sum(prods, Fraction(0))
                exact_abs = sum((abs(p) for p in prods), Fraction(0))
                # S is a sum of non-negative exact fp64 products: relative
                # error at most (K-1)*2^-53 as well.
                bound = Fraction(max(K - 1, 0)) * Fraction(1, 2 ** 53) * exact_abs
                err_c = abs(Fraction(float(C[i, j])) - exact)
                err_s = abs(Fraction(float(S[i, j])) - exact_abs)
                assert err_c <= bound * Fraction(1001, 1000), (
                    f"C[{i},{j}] off by {float(err_c)} > {float(bound)} at {(M, N, K)}")
                assert err_s <= bound * Fraction(1001, 1000), (
                    f"S[{i},{j}] off by {float(err_s)} at {(M, N, K)}")


def pin_identity(gemm: GemmFn, seed: int = 12) -> None:
    rng = np.random.default_rng(seed)
    for M, K in [(1, 1), (7, 5), (33, 17), (64, 64)]:
        A = _rand_f32(rng, (M, K))
        C, _ = gemm(A, np.eye(K, dtype=np.float32))
        assert np.array_equal(C, A.astype(np.float64)), ("A.I", M, K)
        C, _ = gemm(np.eye(M, dtype=np.float32), A)
        assert np.array_equal(C, A.astype(np.float64)), ("I.A", M, K)


def pin_permutation(gemm: GemmFn, seed: int = 13) -> None:
    rng = np.random.default_rng(seed)
    for M, K in [(5, 3), (16, 9), (40, 40)]:
        A = _rand_f32(rng, (M, K))
        pr = rng.permutation(M)
        P = np.zeros((M, M), dtype=np.float32)
        P[np.arange(M), pr] = 1.0           # (P.A)[i] = A[pr[i]]
        C, _ = gemm(P, A)
        assert np.array_equal(C, A[pr].astype(np.float64)), ("P.A", M, K)
        pc = rng.permutation(K)
        Q = np.zeros((K, K), dtype=np.float32)
        Q[pc, np.arange(K)] = 1.0           # (A.Q)[:, j] = A[:, pc[j]]
        C, _ = gemm(A, Q)
        assert np.array_equal(C, A[:, pc].astype(np.float64)), ("A.P", M, K)


def pin_small_integer(gemm: GemmFn, seed: int = 14) -> None:
    rng = np.random.default_rng(seed)
    for M, N, K in [(1, 1, 1), (3, 5, 7), (17, 13, 64), (31, 33, 129)]:
        Ai = rng.integers(-4, 5, size=(M, K))
        Bi = rng.integers(-4, 5, size=(K, N))
        C, S = gemm(Ai.astype(np.float32), Bi.astype(np.float32))
        assert np.array_equal(C, (Ai @ Bi).astype(np.float64)), ("C", M, N, K)
        assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64)), ("S", M, N, K)


def pin_rank_one(gemm: GemmFn, seed: int = 15) -> None:
    rng = np.random.default_rng(seed)
    for M, N, K in [(4, 6, 3), (9, 2, 31), (12, 12, 100)]:
        u = rng.integers(-50, 51, size=M)
        v = rng.integers(-50, 51, size=N)
        A = np.repeat(u[:, None], K, axis=1).astype(np.float32)
        B = np.repeat(v[None, :], K, axis=0).astype(np.float32)
        C, S = gemm(A, B)
        expect = K * np.outer(u, v)
        assert np.array_equal(C, expect.astype(np.float64)), ("rank-1", M, N, K)
        assert np.array_equal(S, np.abs(expect).astype(np.float64)), ("rank-1 S", M, N, K)


def pin_empty(gemm: GemmFn) -> None:
    C, S = gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert C.shape == (3, 4) and not C.any() and not S.any(), "K = 0 must give zeros"
    C, S = gemm(np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))
    assert C.shape == (0, 4)
    C, S = gemm(np.zeros((3, 5), np.float32), np.zeros((5, 0), np.float32))
    assert C.shape == (3, 0)


ALL_PINS = [pin_exact_bound, pin_identity, pin_permutation, pin_small_integer,
            pin_rank_one, pin_empty]


def failing_pins(gemm: GemmFn) -> list:
    """Names of the pins that `gemm` fails (empty when all hold)."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(gemm)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    return failed
