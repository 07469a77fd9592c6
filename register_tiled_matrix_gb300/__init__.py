"""Register-tiled dense product C = A.B for one GB300 (sm_103a).

Two CUDA paths behind a C ABI (include/gemm.h, libgemm_gb300.so):

  gemm_f32      fp32 SIMT kernel: global C tiles, cp.async-staged shared K
                slices, an 8 x 8 fp32 register micro-tile per thread.
  gemm_bf16f32  tcgen05 kernel: TMA-staged bf16 K slices, fp32 accumulators
                in tensor memory, persistent warp-specialised CTAs.

This package is the thin Python binding (torch is used only for device
memory and streams) plus the in-tree build step.
"""

from .native_build import build, ptxas_report  # noqa: F401
from .binding import (  # noqa: F401
    LADDER,
    STATUS,
    GemmError,
    gemm_bf16f32,
    gemm_bf16f32_workspace_bytes,
    gemm_bf16f32_ws,
    gemm_f16f32,
    gemm_f16f32_ws,
    gemm_bf16f32_selftest_timeout,
    gemm_f32,
    gemm_f32_ladder,
    gemm_f32_selftest_timeout,
    gemm_f32_schedule,
    gemm_f32_workspace_bytes,
    F32_KINDS,
    fp32_pipe_peak,
    gemm_f32_ws,
    get_device_error,
    header_symbols,
    library_path,
    load_library,
    status_string,
)
