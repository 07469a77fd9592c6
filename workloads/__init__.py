"""Seeded synthetic inputs for the dense product C = A.B.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds only input generation (shapes, value distributions, seeds,
which output entries to sample) and none of the product's arithmetic.

Every matrix is a contiguous, row-major CPU tensor:
  A is M x K (leading dimension K), B is K x N (leading dimension N).

Value distributions (one per workload):
  "uniform" : i.i.d. uniform on [-1, 1), drawn as 2*U[0,1) - 1 in fp32
  "normal"  : i.i.d. standard normal, fp32
  "int"     : i.i.d. integers uniform in {-4, ..., 4}, stored as fp32
              (every partial sum stays below 2^24, so any summation order
              gives the exact integer result in fp32 and in fp64)
  bf16 workloads draw the fp32 values above and round them to bfloat16
  with round-to-nearest-even (torch's tensor.to(torch.bfloat16)).
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import torch

SEED_BASE = 0x5EED0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # "f32" (gemm_f32) or "bf16" (gemm_bf16f32)
    dist: str           # "uniform" | "normal" | "int"
    seed: int
    full_check: bool    # every entry checked against the oracle, else sampled

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def in_bytes(self) -> int:
        s = 4 if self.dtype == "f32" else 2
        return (self.M * self.K + self.K * self.N) * s

    @property
    def out_bytes(self) -> int:
        return self.M * self.N * 4


def _seed(config_index: int, variant: int = 0) -> int:
    return SEED_BASE + config_index * 16 + variant


# The five configurations of the register-tiled product. Shapes are those of
# the worked examples on the register-tiling pages (64x64 blocks at 1024,
# 128x128 block tiles at 4096) plus ragged shapes and the tensor-core case.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("f32_256_uniform", 256, 256, 256, "f32", "uniform", _seed(1, 0), True),
        Workload("f32_256_int", 256, 256, 256, "f32", "int", _seed(1, 1), True),
        Workload("f32_1024_uniform", 1024, 1024, 1024, "f32", "uniform", _seed(2), True),
        Workload("f32_4096_normal", 4096, 4096, 4096, "f32", "normal", _seed(3), False),
        Workload("f32_1000x1000x999", 1000, 1000, 999, "f32", "uniform", _seed(4, 0), True),
        Workload("f32_4097x3001x1023", 4097, 3001, 1023, "f32", "uniform", _seed(4, 1), False),
        Workload("f32_8192x64x4096", 8192, 64, 4096, "f32", "uniform", _seed(4, 2), True),
        Workload("bf16_8192_normal", 8192, 8192, 8192, "bf16", "normal", _seed(5), False),
        # The tensor-core case with K and N not multiples of 8: no row of A or
        # B starts on a 16-byte boundary after the first.
        Workload("bf16_8192x8190x8190", 8192, 8190, 8190, "bf16", "normal", _seed(5, 1), False),
    ]
}


def _draw(gen: torch.Generator, shape: Tuple[int, int], dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-4, 5, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(M: int, N: int, K: int, dist: str = "uniform", dtype: str = "f32",
                seed: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Return (A, B): A is M x K, B is K x N, contiguous CPU tensors.

    dtype "f32" gives torch.float32; "bf16" gives torch.bfloat16 and "f16"
    torch.float16 (the fp32 draw rounded to nearest even).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    A = _draw(gen, (M, K), dist)
    B = _draw(gen, (K, N), dist)
    if dtype == "bf16":
        A = A.to(torch.bfloat16)
        B = B.to(torch.bfloat16)
    elif dtype == "f16":
        A = A.to(torch.float16)
        B = B.to(torch.float16)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return A.contiguous(), B.contiguous()


def workload_inputs(w: Workload) -> Tuple[torch.Tensor, torch.Tensor]:
    return make_inputs(w.M, w.N, w.K, w.dist, w.dtype, w.seed)


def sample_indices(M: int, N: int, count: int = 4096, seed: int = 0,
                   edge: int = 128, edge_count: int = 64) -> Tuple[torch.Tensor, torch.Tensor]:
    """Seeded (row, col) positions of C to check on large shapes.

    `count` uniform positions, plus the four corners, plus `edge_count`
    positions in the last `edge` rows and as many in the last `edge` columns
    (where ragged tiles end). Returns two int64 tensors of equal length.
    """
    if M <= 0 or N <= 0:
        z = torch.zeros(0, dtype=torch.int64)
        return z, z.clone()
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 1)
    rows: List[torch.Tensor] = [torch.randint(0, M, (count,), generator=gen)]
    cols: List[torch.Tensor] = [torch.randint(0, N, (count,), generator=gen)]
    rows.append(torch.tensor([0, 0, M - 1, M - 1]))
    cols.append(torch.tensor([0, N - 1, 0, N - 1]))
    r0 = max(0, M - edge)
    c0 = max(0, N - edge)
    rows.append(torch.randint(r0, M, (edge_count,), generator=gen))
    cols.append(torch.randint(0, N, (edge_count,), generator=gen))
    rows.append(torch.randint(0, M, (edge_count,), generator=gen))
    cols.append(torch.randint(c0, N, (edge_count,), generator=gen))
    return torch.cat(rows).to(torch.int64), torch.cat(cols).to(torch.int64)
