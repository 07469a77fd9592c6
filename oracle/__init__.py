"""CPU oracle for C = A.B (fp64 accumulation, plain triple loop).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package's smoke check and
by the bench's CPU-baseline leg, never by the product path. It shares no code
with the CUDA library; the only module both sides use is `workloads`, which
draws the seeded inputs.

The arithmetic lives in oracle.c (see its header for the definition followed
and the reading of the pages it takes). This module compiles it with gcc and
calls it through ctypes.

Parity pins: the tests in tests/test_oracle_pins.py check this oracle against
exact rational brute force, identity and permutation matrices, small-integer
products and the closed form of rank-one products, and check that mutated
copies of it (a transposed operand, a dropped term, a flipped sign, an index
off by one) fail those pins.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib: Optional[ctypes.CDLL] = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, a second or so)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded copy of the oracle library."""
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_gemm.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
    lib.oracle_gemm.restype = None
    lib.oracle_gemm_sampled.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p, ctypes.c_int]
    lib.oracle_gemm_sampled.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def _as_f32(x) -> np.ndarray:
    """fp32 C-contiguous numpy copy of a 2-D CPU tensor/array.

    bf16 tensors widen to fp32 exactly (a bf16 value is an fp32 value with
    the low 16 mantissa bits zero)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype != torch.float32:
                x = x.to(torch.float32)
            x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if a.ndim != 2:
        raise ValueError("expected a 2-D matrix")
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gemm(A, B, threads: int = 0, lib: Optional[ctypes.CDLL] = None
         ) -> Tuple[np.ndarray, np.ndarray]:
    """Every entry of C = A.B and of S = sum_k |A[i,k] B[k,j]|, both fp64 M x N.

    `lib` selects another compiled copy of oracle.c (the pin tests pass
    deliberately mutated copies); by default the one built here."""
    a, b = _as_f32(A), _as_f32(B)
    M, K = a.shape
    K2, N = b.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    (lib or _load()).oracle_gemm(M, N, K, a.ctypes.data, b.ctypes.data, C.ctypes.data, S.ctypes.data,
                        int(threads))
    return C, S


def gemm_sampled(A, B, rows, cols, threads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Entries (rows[t], cols[t]) of C and S, as two fp64 vectors."""
    a, b = _as_f32(A), _as_f32(B)
    M, K = a.shape
    K2, N = b.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sampled index outside C")
    Cs = np.empty(r.size, dtype=np.float64)
    Ss = np.empty(r.size, dtype=np.float64)
    _load().oracle_gemm_sampled(M, N, K, a.ctypes.data, b.ctypes.data, r.size, r.ctypes.data,
                                c.ctypes.data, Cs.ctypes.data, Ss.ctypes.data, int(threads))
    return Cs, Ss
