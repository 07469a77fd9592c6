"""CPU tests of the C ABI: the library builds for sm_103a, loads, exports every
symbol that include/gemm.h declares, and rejects bad arguments on the host
before any CUDA call. No kernel is launched here (there is no GPU)."""

import ctypes
import os
import shutil
import subprocess

import pytest

import register_tiled_matrix_gb300 as rtm

pytestmark = pytest.mark.cpu

FAKE = 0x100000  # never dereferenced: every call below returns before any CUDA call


@pytest.fixture(scope="module")
def lib():
    rtm.build()
    return rtm.load_library()


def test_exports_every_declared_symbol(lib):
    names = rtm.header_symbols()
    assert {"gemm_f32", "gemm_f32_ladder", "gemm_f32_ws", "gemm_f32_workspace_bytes",
            "gemm_f32_noalloc", "gemm_bf16f32", "gemm_f16f32", "gemm_get_device_error",
            "gemm_bf16f32_selftest_timeout", "gemm_status_string", "gemm_bf16f32_ws",
            "gemm_f16f32_ws", "gemm_bf16f32_workspace_bytes"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in gemm.h but not exported"


def test_exports_nothing_but_the_entry_points(lib):
    """Built with hidden visibility: the dynamic symbol table holds exactly the
    functions gemm.h declares, so internal C++ names cannot clash with another
    library's in the same process."""
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", rtm.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines()
                if len(line.split()) == 3 and line.split()[1] in "TWVui"}
    assert exported == set(rtm.header_symbols())


def test_status_strings(lib):
    for code, name in rtm.STATUS.items():
        assert rtm.status_string(code).startswith(name)
    assert rtm.status_string(12345) == "unknown gemm status"


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16f32", "gemm_f16f32"])
def test_invalid_sizes(lib, fn):
    f = getattr(lib, fn)
    assert f(-1, 4, 4, FAKE, FAKE, FAKE * 2, None) == -1
    assert f(4, -1, 4, FAKE, FAKE, FAKE * 2, None) == -1
    assert f(4, 4, -8, FAKE, FAKE, FAKE * 2, None) == -1
    assert f(1 << 31, 8, 8, FAKE, FAKE, FAKE * 2, None) == -1


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16f32", "gemm_f16f32"])
def test_empty_output_is_a_noop(lib, fn):
    f = getattr(lib, fn)
    assert f(0, 16, 16, None, None, None, None) == 0
    assert f(16, 0, 16, None, None, None, None) == 0


@pytest.mark.parametrize("fn", ["gemm_f32", "gemm_bf16f32", "gemm_f16f32"])
def test_null_pointers(lib, fn):
    f = getattr(lib, fn)
    assert f(8, 8, 8, FAKE, FAKE, None, None) == -1
    assert f(8, 8, 8, None, FAKE, FAKE * 4, None) == -1
    assert f(8, 8, 8, FAKE, None, FAKE * 4, None) == -1


@pytest.mark.parametrize("fn,elem", [("gemm_f32", 4), ("gemm_bf16f32", 2)])
def test_output_overlapping_input_rejected(lib, fn, elem):
    f = getattr(lib, fn)
    M = N = K = 64
    base = 0x10000000
    assert f(M, N, K, base, base + M * K * elem, base + 16, None) == -1     # C over A
    assert f(M, N, K, base, base + (1 << 20), base + (1 << 20) + 16, None) == -1  # C over B


@pytest.mark.parametrize("fn", ["gemm_bf16f32", "gemm_f16f32"])
def test_tensor_core_alignment_rules(lib, fn):
    """Only pointers off their element size are rejected on the host: any K, N
    and 2-byte-aligned operands are served (by the load-and-swizzle kernel)."""
    f = getattr(lib, fn)
    A, B, C = 0x10000000, 0x20000000, 0x30000000
    assert f(16, 16, 16, A + 1, B, C, None) == -2  # A not 2-byte aligned
    assert f(16, 16, 16, A, B + 3, C, None) == -2
    assert f(16, 16, 16, A, B, C + 2, None) == -2  # C not 4-byte aligned


def test_selftest_needs_k(lib):
    f = lib.gemm_bf16f32_selftest_timeout
    A, B, C = 0x10000000, 0x20000000, 0x30000000
    assert f(16, 16, 0, A, B, C, 10 ** 8, None) == -1  # K == 0 launches no waiting kernel


def test_f32_alignment_rule(lib):
    assert lib.gemm_f32(8, 8, 8, 0x10000001, 0x20000000, 0x30000000, None) == -2


def test_ladder_rung_range(lib):
    f = lib.gemm_f32_ladder
    assert f(-1, 8, 8, 8, FAKE, FAKE, FAKE * 4, None) == -1
    assert f(7, 8, 8, 8, FAKE, FAKE, FAKE * 4, None) == -1
    assert f(1, -8, 8, 8, FAKE, FAKE, FAKE * 4, None) == -1
    assert f(2, 0, 8, 8, None, None, None, None) == 0


def test_workspace_entry_points_host_checks(lib):
    assert lib.gemm_f32_workspace_bytes(-1, 8, 8) == -1
    assert lib.gemm_f32_workspace_bytes(8, 8, 1 << 31) == -1
    assert lib.gemm_f32_workspace_bytes(0, 8, 8) == 0
    assert lib.gemm_f32_workspace_bytes(8, 8, 0) == 0
    f = lib.gemm_f32_ws
    A, B, C, W = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    assert f(8, 8, 8, A, B, C, W, -4, None) == -1        # negative workspace size
    assert f(8, 8, 8, A, B, C, None, 64, None) == -1     # size without a buffer
    assert f(8, 8, 8, A, B, C, W + 2, 64, None) == -2    # misaligned workspace
    assert f(0, 8, 8, None, None, None, None, 0, None) == 0


def test_f32_schedule_host_checks(lib):
    kind, splits = ctypes.c_int(-1), ctypes.c_int(-1)
    f = lib.gemm_f32_schedule
    assert f(-1, 8, 8, 0, ctypes.byref(kind), ctypes.byref(splits)) == -1
    assert f(8, 8, 1 << 31, 1, None, None) == -1
    assert f(0, 8, 8, 0, ctypes.byref(kind), ctypes.byref(splits)) == 0
    assert (kind.value, splits.value) == (0, 1)  # GEMM_F32_NO_KERNEL
    assert f(8, 8, 0, 1, ctypes.byref(kind), None) == 0 and kind.value == 0


def test_f32_schedule_kinds_match_the_header():
    """The binding names exactly the values of gemm_f32_kind in include/gemm.h."""
    import re
    text = open(os.path.join(rtm.native_build.INCLUDE, "gemm.h")).read()
    enum = text[text.index("typedef enum gemm_f32_kind"):text.index("} gemm_f32_kind;")]
    values = {int(v) for v in re.findall(r"GEMM_F32_\w+\s*=\s*(\d+)", enum)}
    assert values == set(rtm.F32_KINDS), (sorted(values), sorted(rtm.F32_KINDS))


def _ceil256(x):
    return (x + 255) // 256 * 256


def test_tensor_core_workspace_size(lib):
    """Room for a copy of A and of B with rows padded to 8 values, each
    rounded up to 256 bytes; none where no re-pitched product would run."""
    f = lib.gemm_bf16f32_workspace_bytes
    for M, N, K in [(300, 129, 77), (129, 1, 1), (8192, 8190, 8190), (4097, 3001, 1023),
                    (256, 256, 256)]:
        expect = _ceil256(M * ((K + 7) // 8 * 8) * 2) + _ceil256(K * ((N + 7) // 8 * 8) * 2)
        assert f(M, N, K) == expect
    assert f(128, 129, 77) == 0
    assert f(300, 0, 77) == 0 and f(300, 129, 0) == 0 and f(0, 129, 77) == 0
    assert f(-1, 8, 8) == -1 and f(300, 8, 1 << 31) == -1


@pytest.mark.parametrize("fn", ["gemm_bf16f32_ws", "gemm_f16f32_ws"])
def test_tensor_core_workspace_host_checks(lib, fn):
    f = getattr(lib, fn)
    A, B, C, W = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    assert f(300, 129, 77, A, B, C, W, -4, None) == -1      # negative workspace size
    assert f(300, 129, 77, A, B, C, None, 64, None) == -1   # size without a buffer
    assert f(300, 129, 77, A + 1, B, C, W, 1 << 20, None) == -2
    assert f(-3, 129, 77, A, B, C, W, 1 << 20, None) == -1
    assert f(0, 129, 77, None, None, None, None, 0, None) == 0


def test_selftest_limit_range(lib):
    f = lib.gemm_bf16f32_selftest_timeout
    A, B, C = 0x10000000, 0x20000000, 0x30000000
    assert f(16, 16, 16, A, B, C, 10, None) == -1
    assert f(16, 16, 16, A, B, C, 10 ** 11, None) == -1


def test_ptxas_zero_spills(lib):
    report = rtm.ptxas_report()
    kernels = list(report)
    assert kernels, "no kernels in the ptxas report"
    for k in kernels:
        r = report[k]
        assert r["spill_stores"] == 0 and r["spill_loads"] == 0, (k, r)
        assert 0 < r["registers"] <= 255, (k, r)
    simt = [report[k] for k in kernels if "sgemm_rt_kernel" in k]
    assert all(r["registers"] <= 128 for r in simt), "two 256-thread CTAs per SM need <= 128 regs"


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """With the library missing, the binding raises instead of computing elsewhere."""
    from register_tiled_matrix_gb300 import binding

    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()
