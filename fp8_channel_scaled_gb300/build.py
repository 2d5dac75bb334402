"""Build the CUDA library in-tree: fp8_channel_scaled_gb300/_lib/libfp8gemm.so.

Each translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked into
one shared library that exports the C ABI of ``include/fp8_gemm.h``.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OBJ_DIR = ROOT / "_build" / "fp8gemm"
LIB_DIR = PKG / "_lib"
LIB = LIB_DIR / "libfp8gemm.so"
SOURCES = ["api.cu", "gemm_tc.cu", "gemm_tc2.cu", "gemm_decode.cu", "repitch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                 "-I", str(INCLUDE), "-I", str(CSRC)]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(home) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def _inputs():
    return [CSRC / s for s in SOURCES] + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + [
        INCLUDE / "fp8_gemm.h"]


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> Path:
    if not force and not extra_flags and up_to_date():
        return LIB
    OBJ_DIR.mkdir(parents=True, exist_ok=True)
    LIB_DIR.mkdir(parents=True, exist_ok=True)
    nv = nvcc()

    def compile_one(src: str):
        obj = OBJ_DIR / (Path(src).stem + ".o")
        cmd = [nv, *CFLAGS, *extra_flags, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB.with_name(f"{LIB.name}.tmp{os.getpid()}")
    # -z defs: an unresolved symbol fails the build instead of the first load
    cmd = [nv, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-Xlinker", "-zdefs", "-o", str(tmp),
           *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=tuple(a for a in sys.argv[1:] if a.startswith("-X")))
    print(LIB)
