"""Helpers for the GPU parity tests: compare a CUDA result with the oracle.

Tolerances (elementwise, S = sum_k |A[i][k] B[k][j]| from the oracle):
  gemm_f32      |C - C_oracle| <= 1e-4 * S
  gemm_bf16f32  |C - C_oracle| <= 1e-3 * S   (oracle fed the same bf16 values)
Where S == 0 the result must be exactly 0. Small-integer inputs, identity and
permutation products must match bit for bit.

Derivation of the fp32 bound's headroom: each output is a sum of K products
formed with fp32 fused multiply-add in some order, so its error is at most
about K * 2^-24 * S in the worst case and ~sqrt(K) * 2^-24 * S typically;
at K = 8192, 2^-24 * 8192 = 4.9e-4 is the pathological worst case while the
typical error (~5e-6 * S) sits far below 1e-4 * S. The tensor-core path
accumulates in fp32 as well; 1e-3 * S leaves room for its internal order.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

TOL = {"f32": 1e-4, "bf16": 1e-3}


def assert_close_to_oracle(C: torch.Tensor, A: torch.Tensor, B: torch.Tensor, dtype: str,
                           full: bool = True, seed: int = 0, count: int = 4096) -> float:
    """Check C (device or host, M x N fp32) against the oracle; return max err/S."""
    tol = TOL[dtype]
    M, N = C.shape
    Ch = C.detach().float().cpu().numpy().astype(np.float64)
    if full:
        C0, S = oracle.gemm(A, B)
        got = Ch
    else:
        rows, cols = workloads.sample_indices(M, N, count=count, seed=seed)
        C0, S = oracle.gemm_sampled(A, B, rows, cols)
        got = Ch[rows.numpy(), cols.numpy()]
    err = np.abs(got - C0)
    assert np.all(np.isfinite(got)), "non-finite output"
    zero = S == 0
    assert np.all(got[zero] == 0), "entries with an all-zero product sum must be exactly 0"
    ratio = np.where(zero, 0.0, err / np.where(zero, 1.0, S))
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = np.argwhere(ratio > tol)
    assert bad.size == 0, (
        f"{bad.shape[0]} entries exceed {tol}*S; worst err/S = {worst:.3e} at {bad[0].tolist()}")
    return worst


def assert_bit_exact(C: torch.Tensor, expect) -> None:
    got = C.detach().float().cpu()
    exp = torch.as_tensor(np.asarray(expect), dtype=torch.float32)
    assert got.shape == exp.shape
    diff = (got != exp).nonzero()
    assert diff.numel() == 0, f"{diff.shape[0]} entries differ, first at {diff[0].tolist()}"


def small_int_inputs(M: int, N: int, K: int, seed: int):
    return workloads.make_inputs(M, N, K, "int", "f32", seed=seed)


def guarded_output(M: int, N: int, device, pad: int = 4096, sentinel: float = float("nan")):
    """An M x N output view inside a buffer padded by `pad` floats on each side."""
    buf = torch.full((pad + M * N + pad,), sentinel, dtype=torch.float32, device=device)
    return buf, buf[pad:pad + M * N].view(M, N)


def guard_intact(buf: torch.Tensor, M: int, N: int, pad: int = 4096) -> bool:
    head = buf[:pad]
    tail = buf[pad + M * N:]
    return bool(torch.isnan(head).all().item() and torch.isnan(tail).all().item())


def kernel_names(fn) -> list:
    """Names of the kernels one call of fn launches (profiler kernel records;
    the first session of a process may start its tracer after the launches,
    so sessions repeat until one records any)."""
    from torch.profiler import ProfilerActivity, profile

    for _ in range(3):
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events()
                 if str(getattr(e, "device_type", "")).endswith("CUDA")
                 and not e.name.startswith(("Memcpy", "Memset"))]
        if names:
            return names
    return names
