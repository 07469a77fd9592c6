"""Several host threads make their first calls into a freshly loaded library at
once, each on its own stream: the per-device caches filled on first use (SM
count, driver entry point, kernel attributes, cluster occupancy) must come out
right whichever thread gets there first. Runs in a child process so that the
library's first use really happens inside the threads."""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    import numpy as np
    import torch
    import register_tiled_matrix_gb300 as rtm
    import workloads, oracle

    torch.cuda.init()
    jobs = []
    for i in range(12):
        kind = ["f32", "f32_ws", "bf16", "bf16_small", "f16", "bf16_ws", "bf16_any", "f32",
                "f32", "bf16_any", "bf16_any", "f32_ws"][i]
        M, N, K = [(300, 260, 129), (256, 64, 2048), (384, 264, 200), (96, 1024, 136),
                   (300, 264, 72), (300, 129, 77), (120, 100, 33), (1000, 1000, 999),
                   (2000, 60, 2000),
                   (64, 1030, 4098),    # transposed load-and-swizzle, K split over 4
                   (1000, 120, 2052),   # the same without the swap (tall, narrow)
                   (640, 518, 2047)][i]  # fp32 operands re-pitched into the workspace
        dt = {"f32": "f32", "f32_ws": "f32", "f16": "f16"}.get(kind, "bf16")
        A, B = workloads.make_inputs(M, N, K, "normal", dt, seed=i + 11)
        jobs.append((kind, A, B))

    fns = {"f32": rtm.gemm_f32, "f32_ws": rtm.gemm_f32_ws, "bf16": rtm.gemm_bf16f32,
           "bf16_small": rtm.gemm_bf16f32, "f16": rtm.gemm_f16f32, "bf16_ws": rtm.gemm_bf16f32_ws,
           "bf16_any": rtm.gemm_bf16f32}
    dev = [(kind, A.cuda(), B.cuda()) for kind, A, B in jobs]
    streams = [torch.cuda.Stream() for _ in jobs]
    torch.cuda.synchronize()
    results = [None] * len(jobs)
    errors = []
    barrier = threading.Barrier(len(jobs))

    def work(i):
        try:
            kind, A, B = dev[i]
            barrier.wait()
            with torch.cuda.stream(streams[i]):
                for _ in range(3):
                    C = fns[kind](A, B, stream=streams[i])
            streams[i].synchronize()
            results[i] = C.cpu()
        except Exception as e:  # reported by the parent
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        print("\n".join(errors)); sys.exit(2)
    if rtm.get_device_error() != 0:
        print("device error word set"); sys.exit(3)
    for (kind, A, B), C in zip(jobs, results):
        C0, S = oracle.gemm(A, B)
        tol = 1e-4 if kind.startswith("f32") else 1e-3
        err = np.abs(C.double().numpy() - C0)
        if not np.all(err <= tol * S):
            print(f"{kind}: max err/S {float((err / np.maximum(S, 1e-300)).max()):.3e}"); sys.exit(4)
    print("ok")
""")


def test_first_calls_from_many_threads():
    import register_tiled_matrix_gb300 as rtm
    rtm.build()  # build in this process; the child only loads the library
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
