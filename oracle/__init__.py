"""CPU oracle for the per-output-channel scaled FP8 linear layer.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg are the only users of this package; the CUDA
library and its Python binding never import, load or call it, and it never
imports them.

The arithmetic lives in ``oracle.c`` (plain C, POSIX threads): an E4M3FN
decode table built from the bit fields, exact fp64 dot products, one
multiplication by the fp32 per-output-channel scale and one round-to-
nearest-even to bf16.  This module only compiles that file (``build``) and
marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if not force and _LIB.exists() and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L",
           "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(str(build()))
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_e4m3_table.argtypes = [f64p]
    lib.oracle_e4m3_table.restype = None
    lib.oracle_bf16_of_product.argtypes = [ctypes.c_double, ctypes.c_float]
    lib.oracle_bf16_of_product.restype = ctypes.c_uint16
    lib.oracle_dot.argtypes = [u8p, u8p, i64, i64, i64, f64p, ctypes.c_int]
    lib.oracle_linear.argtypes = [u8p, u8p, f32p, i64, i64, i64, u16p, ctypes.c_int]
    lib.oracle_linear_rows.argtypes = [u8p, u8p, f32p, i64, i64, i64, i64p, i64,
                                       u16p, ctypes.c_int]
    lib.oracle_linear_elems.argtypes = [u8p, u8p, f32p, i64, i64, i64, i64p, i64,
                                        u16p, ctypes.c_int]
    for f in ("oracle_dot", "oracle_linear", "oracle_linear_rows", "oracle_linear_elems"):
        getattr(lib, f).restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    lib.oracle_default_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _operands(x, w, scale):
    x = np.ascontiguousarray(x, dtype=np.uint8)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"bad operand shapes {x.shape} {w.shape}")
    if scale is not None:
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        if scale.shape != (w.shape[0],):
            raise ValueError(f"scale shape {scale.shape} != ({w.shape[0]},)")
    return x, w, scale


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 E4M3FN codes (NaN for 0x7F and 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out, ctypes.c_double))
    return out


def bf16_of_product(d: float, s: float) -> int:
    """bf16 bit pattern of RNE(d * s) with d a double and s an fp32, rounded once."""
    return int(_load().oracle_bf16_of_product(float(d), float(np.float32(s))))


def dot(x, w, nthreads: int = 0) -> np.ndarray:
    """Exact fp64 dot products d[m, n] = sum_k dec(x[m,k]) * dec(w[n,k])."""
    x, w, _ = _operands(x, w, None)
    M, K = x.shape
    N = w.shape[0]
    d = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_dot(_ptr(x, ctypes.c_uint8), _ptr(w, ctypes.c_uint8),
                              M, N, K, _ptr(d, ctypes.c_double), nthreads), "dot")
    return d


def linear(x, w, scale, nthreads: int = 0) -> np.ndarray:
    """All outputs y[M, N] as bf16 bit patterns (uint16)."""
    x, w, scale = _operands(x, w, scale)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), dtype=np.uint16)
    _check(_load().oracle_linear(_ptr(x, ctypes.c_uint8), _ptr(w, ctypes.c_uint8),
                                 _ptr(scale, ctypes.c_float), M, N, K,
                                 _ptr(y, ctypes.c_uint16), nthreads), "linear")
    return y


def linear_rows(x, w, scale, rows, nthreads: int = 0) -> np.ndarray:
    """Outputs of the listed rows only: y[len(rows), N] bf16 bit patterns."""
    x, w, scale = _operands(x, w, scale)
    M, K = x.shape
    N = w.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    y = np.empty((rows.size, N), dtype=np.uint16)
    _check(_load().oracle_linear_rows(_ptr(x, ctypes.c_uint8), _ptr(w, ctypes.c_uint8),
                                      _ptr(scale, ctypes.c_float), M, N, K,
                                      _ptr(rows, ctypes.c_int64), rows.size,
                                      _ptr(y, ctypes.c_uint16), nthreads), "linear_rows")
    return y


def linear_elems(x, w, scale, rows, cols, nthreads: int = 0) -> np.ndarray:
    """Outputs y[rows[i], cols[i]] as bf16 bit patterns."""
    x, w, scale = _operands(x, w, scale)
    M, K = x.shape
    N = w.shape[0]
    rc = np.ascontiguousarray(np.stack([np.asarray(rows, np.int64),
                                        np.asarray(cols, np.int64)], axis=1))
    y = np.empty(rc.shape[0], dtype=np.uint16)
    _check(_load().oracle_linear_elems(_ptr(x, ctypes.c_uint8), _ptr(w, ctypes.c_uint8),
                                       _ptr(scale, ctypes.c_float), M, N, K,
                                       _ptr(rc, ctypes.c_int64), rc.shape[0],
                                       _ptr(y, ctypes.c_uint16), nthreads), "linear_elems")
    return y


def default_threads() -> int:
    """Threads a call with nthreads=0 uses (all online host cores)."""
    return int(_load().oracle_default_threads())


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
