"""ctypes binding of libgemm_gb300.so: argument marshalling only.

Every step of the product runs in the library's CUDA kernels; this module
checks tensor metadata, allocates the output with torch when the caller gives
none, passes raw device pointers and the current torch stream, and turns a
non-zero status into an exception. There is no CPU fallback: if the library
is missing the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Tuple

import torch

from . import native_build as _build

STATUS = {
    0: "GEMM_OK",
    -1: "GEMM_ERR_INVALID_ARG",
    -2: "GEMM_ERR_ALIGNMENT",
    -3: "GEMM_ERR_LAUNCH",
    -4: "GEMM_ERR_TIMEOUT",
    -5: "GEMM_ERR_DEVICE",
}

_lib: Optional[ctypes.CDLL] = None


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Load the built library (build it first with register_tiled_matrix_gb300.build())."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is not built: call register_tiled_matrix_gb300.build() "
                "(nvcc, sm_103a) first; there is no fallback implementation")
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        for name in ("gemm_f32", "gemm_bf16f32", "gemm_f16f32"):
            f = getattr(lib, name)
            f.argtypes = [i64, i64, i64, p, p, p, p]
            f.restype = ctypes.c_int
        lib.gemm_f32_workspace_bytes.argtypes = [i64, i64, i64]
        lib.gemm_f32_workspace_bytes.restype = ctypes.c_int64
        lib.gemm_f32_schedule.argtypes = [i64, i64, i64, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.gemm_f32_schedule.restype = ctypes.c_int
        lib.gemm_f32_ws.argtypes = [i64, i64, i64, p, p, p, p, i64, p]
        lib.gemm_f32_ws.restype = ctypes.c_int
        lib.gemm_bf16f32_workspace_bytes.argtypes = [i64, i64, i64]
        lib.gemm_bf16f32_workspace_bytes.restype = ctypes.c_int64
        for name in ("gemm_bf16f32_ws", "gemm_f16f32_ws"):
            f = getattr(lib, name)
            f.argtypes = [i64, i64, i64, p, p, p, p, i64, p]
            f.restype = ctypes.c_int
        lib.gemm_f32_ladder.argtypes = [ctypes.c_int, i64, i64, i64, p, p, p, p]
        lib.gemm_f32_ladder.restype = ctypes.c_int
        lib.gemm_bf16f32_selftest_timeout.argtypes = [i64, i64, i64, p, p, p, i64, p]
        lib.gemm_bf16f32_selftest_timeout.restype = ctypes.c_int
        lib.gemm_f32_selftest_timeout.argtypes = [i64, i64, i64, p, p, p, i64, p]
        lib.gemm_f32_selftest_timeout.restype = ctypes.c_int
        lib.gemm_fp32_pipe_peak.argtypes = [i64, ctypes.c_int, p, ctypes.POINTER(ctypes.c_double),
                                            p]
        lib.gemm_fp32_pipe_peak.restype = ctypes.c_int
        lib.gemm_get_device_error.argtypes = [p]
        lib.gemm_get_device_error.restype = ctypes.c_int
        lib.gemm_status_string.argtypes = [ctypes.c_int]
        lib.gemm_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def header_symbols() -> List[str]:
    """Names of the functions declared in include/gemm.h."""
    path = os.path.join(_build.INCLUDE, "gemm.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def _check(status: int) -> None:
    if status != 0:
        raise GemmError(status, status_string(status))


# The current stream's handle without building a torch.cuda.Stream object
# (about a microsecond per call); the public API where the accessor is absent.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream: Optional[torch.cuda.Stream], device: Optional[int] = None) -> int:
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_current_stream is not None:
        return int(_raw_current_stream(torch.cuda.current_device() if device is None else device))
    return int(torch.cuda.current_stream().cuda_stream)


class _SameDevice:
    """The device guard of a call whose tensors are on the current device: none."""

    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_SAME_DEVICE = _SameDevice()


def _on_device(t: torch.Tensor):
    """A context that makes t's device current for the call (switching only when
    it is not current already: the switch and switch back cost microseconds)."""
    idx = t.get_device()
    return _SAME_DEVICE if idx == torch.cuda.current_device() else torch.cuda.device(idx)


def _library() -> ctypes.CDLL:
    return _lib if _lib is not None else load_library()


def _prepare(A: torch.Tensor, B: torch.Tensor, dtype: torch.dtype,
             out: Optional[torch.Tensor]) -> torch.Tensor:
    for name, t in (("A", A), ("B", B)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D (row-major) matrix")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {M}x{K}, B is {K2}x{N}")
    if A.device != B.device:
        raise ValueError("A and B must be on the same device")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif (out.dtype != torch.float32 or out.shape != (M, N) or not out.is_contiguous()
          or out.device != A.device):
        raise ValueError("out must be a contiguous float32 M x N tensor on A's device")
    return out


def gemm_f32(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B on the SIMT FP32 register-tiled kernel (fp32 in, fp32 out)."""
    C = _prepare(A, B, torch.float32, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(_library().gemm_f32(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                       _stream_handle(stream, A.get_device())))
    return C


F32_KINDS = {0: "none", 1: "tiles", 2: "tiles+cluster-split", 3: "tiles+workspace-split",
             4: "column-strips", 5: "tiles+tail-cluster-split", 6: "tall-tiles",
             7: "tall-tiles+cluster-split", 8: "wide-tiles", 9: "wide-tiles+cluster-split",
             10: "tiles+stream-k"}


def gemm_f32_schedule(M: int, N: int, K: int, workspace: bool = False) -> Tuple[str, int]:
    """(kind, splits): how gemm_f32 (or gemm_f32_ws, workspace=True) computes this
    shape on the current device; kind is a value of F32_KINDS."""
    kind, splits = ctypes.c_int(-1), ctypes.c_int(0)
    _check(load_library().gemm_f32_schedule(int(M), int(N), int(K), 1 if workspace else 0,
                                            ctypes.byref(kind), ctypes.byref(splits)))
    return F32_KINDS[kind.value], splits.value


def gemm_f32_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes gemm_f32_ws uses for this shape on the current device (0: none)."""
    n = int(load_library().gemm_f32_workspace_bytes(int(M), int(N), int(K)))
    _check(n if n < 0 else 0)
    return n


def gemm_f32_ws(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B, splitting K over a workspace when the shape has too few C tiles.

    `workspace` is a CUDA tensor of at least gemm_f32_workspace_bytes(M, N, K)
    bytes; when None, one is allocated with torch for this call."""
    C = _prepare(A, B, torch.float32, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        if workspace is None:
            need = gemm_f32_workspace_bytes(M, N, K)
            workspace = torch.empty(max(need // 4, 1), dtype=torch.float32, device=A.device)
        if not workspace.is_cuda or workspace.device != A.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor on A's device")
        nbytes = workspace.numel() * workspace.element_size()
        _check(_library().gemm_f32_ws(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                      workspace.data_ptr(), nbytes,
                                      _stream_handle(stream, A.get_device())))
    return C


LADDER = {0: "naive", 1: "shared-tiled 32x32", 2: "register-tiled 64x64, 4x4/thread",
          3: "register-tiled 128x128, 8x8/thread (gemm_f32)",
          4: "register-tiled 16x16, 1x1/thread (rung 2's kernel, T=1)",
          5: "register-tiled 32x32, 2x2/thread (rung 2's kernel, T=2)",
          6: "register-tiled 128x128, 8x8/thread (rung 2's kernel, T=8)"}


def gemm_f32_ladder(rung: int, A: torch.Tensor, B: torch.Tensor,
                    out: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B with rung `rung` of the page's ablation ladder (see LADDER)."""
    C = _prepare(A, B, torch.float32, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(load_library().gemm_f32_ladder(int(rung), M, N, K, A.data_ptr(), B.data_ptr(),
                                              C.data_ptr(), _stream_handle(stream, A.get_device())))
    return C


def gemm_bf16f32(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B on the tcgen05 tensor-core kernel (bf16 in, fp32 accumulate and out)."""
    C = _prepare(A, B, torch.bfloat16, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(_library().gemm_bf16f32(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                           _stream_handle(stream, A.get_device())))
    return C


def gemm_f16f32(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B on the tcgen05 tensor-core kernel (fp16 in, fp32 accumulate and out)."""
    C = _prepare(A, B, torch.float16, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(_library().gemm_f16f32(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                          _stream_handle(stream, A.get_device())))
    return C


def gemm_bf16f32_workspace_bytes(M: int, N: int, K: int) -> int:
    """Largest workspace gemm_bf16f32_ws / gemm_f16f32_ws may use for this shape (0: none)."""
    n = int(load_library().gemm_bf16f32_workspace_bytes(int(M), int(N), int(K)))
    _check(n if n < 0 else 0)
    return n


def _rows_on_16_bytes(t: torch.Tensor) -> bool:
    return t.shape[1] % 8 == 0 and t.data_ptr() % 16 == 0


def _gemm_2byte_ws(entry: str, A: torch.Tensor, B: torch.Tensor, dtype: torch.dtype,
                   out: Optional[torch.Tensor], workspace: Optional[torch.Tensor],
                   stream: Optional[torch.cuda.Stream]) -> torch.Tensor:
    C = _prepare(A, B, dtype, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        if workspace is None and M > 128 and not (_rows_on_16_bytes(A) and _rows_on_16_bytes(B)):
            workspace = torch.empty(gemm_bf16f32_workspace_bytes(M, N, K), dtype=torch.uint8,
                                    device=A.device)
        ptr, nbytes = 0, 0
        if workspace is not None:
            if (not workspace.is_cuda or workspace.device != A.device
                    or not workspace.is_contiguous()):
                raise ValueError("workspace must be a contiguous CUDA tensor on A's device")
            ptr, nbytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        _check(getattr(_library(), entry)(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                          ptr, nbytes, _stream_handle(stream, A.get_device())))
    return C


def gemm_bf16f32_ws(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """gemm_bf16f32, re-pitching operands whose rows are not 16-byte aligned into
    `workspace` (a CUDA tensor of at least gemm_bf16f32_workspace_bytes(M, N, K)
    bytes; allocated with torch for this call when None and a copy is needed)."""
    return _gemm_2byte_ws("gemm_bf16f32_ws", A, B, torch.bfloat16, out, workspace, stream)


def gemm_f16f32_ws(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """gemm_f16f32 with the workspace rule of gemm_bf16f32_ws."""
    return _gemm_2byte_ws("gemm_f16f32_ws", A, B, torch.float16, out, workspace, stream)


def gemm_bf16f32_selftest_timeout(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor,
                                  wait_limit_ns: int,
                                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the bf16 kernel with its loads muted so every bounded wait runs out."""
    C = _prepare(A, B, torch.bfloat16, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(load_library().gemm_bf16f32_selftest_timeout(
            M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), int(wait_limit_ns),
            _stream_handle(stream)))


def gemm_f32_selftest_timeout(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor,
                              wait_limit_ns: int,
                              stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch gemm_f32's TMA-fed kernel with its loads muted so every bounded wait runs out."""
    C = _prepare(A, B, torch.float32, out)
    M, K = A.shape
    N = B.shape[1]
    with _on_device(A):
        _check(load_library().gemm_f32_selftest_timeout(
            M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), int(wait_limit_ns),
            _stream_handle(stream)))


def get_device_error(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream; return and clear the device error word."""
    return int(load_library().gemm_get_device_error(_stream_handle(stream)))


def fp32_pipe_peak(iters: int = 20000, packed: bool = False, repeats: int = 5,
                   device: Optional[torch.device] = None) -> dict:
    """Measured throughput of the FP32 FMA pipes (gemm_fp32_pipe_peak).

    Times `repeats` launches with CUDA events on the current stream after one
    warm-up launch and returns the best: {"tflops", "ms", "sm_mhz"} where
    sm_mhz is the SM clock the launch ran at (clock cycles over global-timer
    nanoseconds, read by the kernel)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    lib = load_library()
    best = None
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        clk = torch.zeros(2, dtype=torch.int64, device=dev)
        flops = ctypes.c_double(0.0)
        for r in range(repeats + 1):
            clk.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _check(lib.gemm_fp32_pipe_peak(int(iters), 1 if packed else 0, clk.data_ptr(),
                                           ctypes.byref(flops), int(stream.cuda_stream)))
            e1.record(stream)
            stream.synchronize()
            if r == 0:
                continue  # warm-up launch
            ms = e0.elapsed_time(e1)
            cycles, ns = (int(v) for v in clk.cpu().tolist())
            res = {"tflops": flops.value / (ms * 1e-3) / 1e12, "ms": ms,
                   "sm_mhz": (cycles / ns * 1e3) if ns > 0 else None}
            if best is None or res["tflops"] > best["tflops"]:
                best = res
    return best
