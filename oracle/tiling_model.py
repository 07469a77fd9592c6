"""Counting model of the kernels the register-tiling page compares.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/): used by tests/ and by the
bench's ablation-ladder report, never by the product path.

"【infra之路】理解 Register Tiling" walks from a kernel that reads global
memory directly, to a shared-memory tiled kernel (one output per thread), to a
register-tiled kernel (a 4 x 4 block of outputs per thread), and accounts for
the reads each one makes (sections "先看 Shared Memory 版本里，一个线程在做什么",
"Register Tiling 的核心思想", "关键循环：为什么省了 Shared Memory 读取？" and
"用一张图对比三个版本"). This module runs those loops literally, on the CPU,
with one counter per memory level, and computes C in fp64 along the way:

  * the product it returns must equal the plain definition (the oracle), since
    tiling only re-groups the sum over k;
  * the counters reproduce the numbers the page prints (tests/golden/).

Pure-Python loops: small shapes only (a few times 64^3 multiply-adds).

Readings of the page (its code leaves these open): the shared kernel uses
TILE x TILE threads with one output each; the register kernel uses 16 x 16
threads, TM = TN = 4, thread (ty, tx) owns rows ty*TM .. +TM-1 and columns
tx*TN .. +TN-1 (threadRow, threadCol of the page's loop), the K-slice depth BK
is a free parameter, and the cooperative global->shared load reads every
element of the A and B slices exactly once per block. Out-of-range elements
are loaded as zeros and not counted as reads.
"""

from __future__ import annotations

import dataclasses
from typing import Tuple

import numpy as np


@dataclasses.dataclass
class Counts:
    global_reads: int = 0   # 4-byte elements read from global memory
    shared_reads: int = 0   # 4-byte elements read from shared memory
    fmas: int = 0           # multiply-adds

    def per_output(self, M: int, N: int) -> dict:
        return {"global": self.global_reads / (M * N), "shared": self.shared_reads / (M * N),
                "fmas": self.fmas / (M * N)}


def _shape(A, B):
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    return A, B, M, N, K


def naive(A, B) -> Tuple[np.ndarray, Counts]:
    """One thread per output; every operand straight from global memory."""
    A, B, M, N, K = _shape(A, B)
    C = np.zeros((M, N))
    c = Counts()
    for row in range(M):
        for col in range(N):
            s = 0.0
            for k in range(K):
                s += A[row, k] * B[k, col]
                c.global_reads += 2
                c.fmas += 1
            C[row, col] = s
    return C, c


def shared_tiled(A, B, tile: int = 32) -> Tuple[np.ndarray, Counts]:
    """TILE x TILE threads, one output each; A and B tiles staged in shared memory."""
    A, B, M, N, K = _shape(A, B)
    C = np.zeros((M, N))
    c = Counts()
    for by in range(0, M, tile):
        for bx in range(0, N, tile):
            acc = np.zeros((tile, tile))
            for k0 in range(0, K, tile):
                # cooperative load: thread (ty, tx) copies sA[ty][tx] and sB[ty][tx]
                sA = np.zeros((tile, tile))
                sB = np.zeros((tile, tile))
                for ty in range(tile):
                    for tx in range(tile):
                        if by + ty < M and k0 + tx < K:
                            sA[ty, tx] = A[by + ty, k0 + tx]
                            c.global_reads += 1
                        if k0 + ty < K and bx + tx < N:
                            sB[ty, tx] = B[k0 + ty, bx + tx]
                            c.global_reads += 1
                # compute: sum += sA[ty][k] * sB[k][tx]
                for ty in range(tile):
                    for tx in range(tile):
                        if by + ty >= M or bx + tx >= N:
                            continue
                        s = acc[ty, tx]
                        for k in range(tile):
                            s += sA[ty, k] * sB[k, tx]
                            c.shared_reads += 2
                            c.fmas += 1
                        acc[ty, tx] = s
            for ty in range(tile):
                for tx in range(tile):
                    if by + ty < M and bx + tx < N:
                        C[by + ty, bx + tx] = acc[ty, tx]
    return C, c


def register_tiled(A, B, threads: int = 16, TM: int = 4, TN: int = 4,
                   BK: int = 16) -> Tuple[np.ndarray, Counts]:
    """threads x threads threads, a TM x TN output block each (the page's loop)."""
    A, B, M, N, K = _shape(A, B)
    BM, BN = threads * TM, threads * TN
    C = np.zeros((M, N))
    c = Counts()
    for by in range(0, M, BM):
        for bx in range(0, N, BN):
            results = np.zeros((threads, threads, TM, TN))  # threadResults per thread
            for k0 in range(0, K, BK):
                sA = np.zeros((BM, BK))
                sB = np.zeros((BK, BN))
                for r in range(BM):
                    for kk in range(BK):
                        if by + r < M and k0 + kk < K:
                            sA[r, kk] = A[by + r, k0 + kk]
                            c.global_reads += 1
                for kk in range(BK):
                    for col in range(BN):
                        if k0 + kk < K and bx + col < N:
                            sB[kk, col] = B[k0 + kk, bx + col]
                            c.global_reads += 1
                for ty in range(threads):
                    for tx in range(threads):
                        thread_row, thread_col = ty * TM, tx * TN
                        # a thread whose whole block lies outside C does no work
                        if by + thread_row >= M or bx + thread_col >= N:
                            continue
                        res = results[ty, tx]
                        for k in range(BK):
                            regA = [sA[thread_row + m, k] for m in range(TM)]
                            regB = [sB[k, thread_col + n] for n in range(TN)]
                            c.shared_reads += TM + TN
                            for m in range(TM):
                                for n in range(TN):
                                    res[m, n] += regA[m] * regB[n]
                                    c.fmas += 1
            for ty in range(threads):
                for tx in range(threads):
                    for m in range(TM):
                        for n in range(TN):
                            r, col = by + ty * TM + m, bx + tx * TN + n
                            if r < M and col < N:
                                C[r, col] = results[ty, tx, m, n]
    return C, c


def predicted_shared_reads_per_output_per_k(TM: int, TN: int) -> float:
    """Shared reads per output per k of a TM x TN register tile: (TM + TN) / (TM TN)."""
    return (TM + TN) / (TM * TN)


def predicted_global_reads_per_output(K: int, BM: int, BN: int) -> float:
    """Global reads per output of a BM x BN block tile staged once per K-slice."""
    return K * (BM + BN) / (BM * BN)
