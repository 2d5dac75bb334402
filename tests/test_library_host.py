"""Host-side checks of the CUDA library: it builds, loads, exports the C ABI,
and rejects bad arguments before touching a GPU.  No compute calls."""
import ast
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8_gemm.h")
PKG = os.path.join(ROOT, "fp8_channel_scaled_gb300")


@pytest.fixture(scope="module")
def cdll():
    from fp8_channel_scaled_gb300 import build
    build.build()
    import fp8_channel_scaled_gb300 as f
    return f.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_gemm_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("fp8_gemm_scaled", "fp8_gemm_scaled_ex", "fp8_gemm_plan",
              "fp8_gemm_check_device_error", "fp8_gemm_status_string", "fp8_gemm_version",
              "fp8_gemm_selftest_wait_timeout", "fp8_gemm_set_wait_budget_ns"):
        assert n in names


def test_library_exports_every_declared_symbol(cdll):
    lib_path = cdll._name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\S+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(cdll, n)


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_version_and_status_strings(cdll):
    import fp8_channel_scaled_gb300 as f
    assert f.fp8_gemm_version() == 6
    for s in range(9):
        assert f.fp8_gemm_status_string(s) and f.fp8_gemm_status_string(s) != "unknown status"
    assert f.fp8_gemm_status_string(99) == "unknown status"


def test_argument_checks_before_any_cuda_call(cdll):
    vp = ctypes.c_void_p
    # negative sizes and null pointers are rejected on the host
    assert cdll.fp8_gemm_scaled(None, None, None, None, -1, 4, 4, None) == 1
    assert cdll.fp8_gemm_scaled(None, None, None, None, 4, 4, 4, None) == 1
    # empty problems are a no-op
    assert cdll.fp8_gemm_scaled(None, None, None, None, 0, 4, 4, None) == 0
    assert cdll.fp8_gemm_scaled(None, None, None, None, 4, 0, 4, None) == 0
    # misaligned scale / y
    assert cdll.fp8_gemm_scaled(vp(16), vp(16), vp(18), vp(1024), 4, 4, 4, None) == 2
    assert cdll.fp8_gemm_scaled(vp(16), vp(16), vp(32), vp(1025), 4, 4, 4, None) == 2
    # y overlapping x
    assert cdll.fp8_gemm_scaled(vp(4096), vp(1 << 20), vp(1 << 22), vp(4096 + 8), 4, 4, 4, None) == 1
    # non-zero reserved option fields
    import fp8_channel_scaled_gb300._binding as b
    o = b._COptions()
    o.reserved = 7
    assert cdll.fp8_gemm_plan(0, None, None, 4, 4, 4, ctypes.byref(o), ctypes.byref(b._CPlan())) in (1, 3)


def test_product_path_never_touches_the_oracle():
    """The package and the CUDA sources neither import nor name oracle/."""
    for dirpath, _, files in os.walk(PKG):
        for fn in files:
            if not fn.endswith((".py", ".cu", ".cuh", ".h")):
                continue
            text = open(os.path.join(dirpath, fn)).read()
            if fn.endswith(".py"):
                tree = ast.parse(text)
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert not any(a.name.split(".")[0] in ("oracle", "synth") for a in node.names), fn
                    if isinstance(node, ast.ImportFrom):
                        assert (node.module or "").split(".")[0] not in ("oracle", "synth"), fn
            else:
                assert "oracle" not in text.lower(), fn


def test_binding_fails_loudly_without_library(tmp_path):
    """With the shared library absent, the binding raises instead of falling back."""
    code = (
        "import fp8_channel_scaled_gb300._binding as b, pathlib\n"
        f"b._LIB_PATH = pathlib.Path({str(tmp_path)!r}) / 'missing.so'\n"
        "try:\n"
        "    b.lib()\n"
        "except b.FP8GemmError as e:\n"
        "    print('raised', e.status)\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert "raised 3" in r.stdout, r.stdout + r.stderr


def test_oracle_and_library_share_no_code():
    osrc = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert "#include \"" not in osrc  # only system headers
    for fn in os.listdir(os.path.join(PKG, "csrc")):
        text = open(os.path.join(PKG, "csrc", fn)).read()
        assert "oracle" not in text.lower()
