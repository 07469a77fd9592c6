"""Compile the CUDA library libgemm_gb300.so in-tree for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/ (with -Xptxas -v; the register/spill report is kept in
_build/ptxas.log), then linked into a shared library next to this file.
Rebuilds only when a source or header is newer than the library.
"""

from __future__ import annotations

import concurrent.futures
import os
import re
import shutil
import subprocess
from typing import Dict, List

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgemm_gb300.so")
PTXAS_LOG = os.path.join(BUILD, "ptxas.log")

SOURCES = ["api.cu", "sgemm_simt.cu", "sgemm_ladder.cu", "gemm_tc.cu", "gemm_tc2.cu",
           "gemm_tc_any.cu", "noalloc.cu", "pack.cu", "sgemm_plan.cu", "tc_plan.cu",
           "gemm_tc_t.cu", "sgemm_short.cu", "fp32_peak.cu", "sgemm_tma.cu",
           "sgemm_tma_rect.cu", "gemm_tc_any_t.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return path


def _inputs() -> List[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Build (if needed) and return the path of libgemm_gb300.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(_compile, SOURCES))
    with open(PTXAS_LOG, "w") as f:
        for src, log in zip(SOURCES, logs):
            f.write(f"==== {src}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(PTXAS_LOG).read())
    return LIB


def ptxas_report() -> Dict[str, Dict[str, int]]:
    """Per-kernel registers, spill bytes and shared memory from the last build."""
    out: Dict[str, Dict[str, int]] = {}
    if not os.path.exists(PTXAS_LOG):
        return out
    current = None
    for line in open(PTXAS_LOG):
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            current = m.group(1)
            out[current] = {"registers": -1, "spill_stores": 0, "spill_loads": 0, "smem": 0}
            continue
        if current is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            out[current]["spill_stores"] = int(m.group(1))
            out[current]["spill_loads"] = int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            out[current]["registers"] = int(m.group(1))
            m2 = re.search(r"(\d+) bytes smem", line)
            if m2:
                out[current]["smem"] = int(m2.group(1))
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
