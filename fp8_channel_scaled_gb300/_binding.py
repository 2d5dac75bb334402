"""ctypes marshalling for include/fp8_gemm.h.  No computation happens here."""
from __future__ import annotations

import ctypes
import dataclasses
import threading
from dataclasses import dataclass
from pathlib import Path

_PKG = Path(__file__).resolve().parent
_LIB_PATH = _PKG / "_lib" / "libfp8gemm.so"

PATH_AUTO, PATH_MAIN, PATH_DECODE = 0, 1, 2
STATUS = {0: "OK", 1: "EINVAL", 2: "EALIGN", 3: "EDEVICE", 4: "ELAUNCH", 5: "ETIMEOUT",
          6: "EUNSUPPORTED", 7: "ESIZE", 8: "ENOMEM"}
NOALLOC_WORKSPACE_BYTES = 32 * 1024 * 1024


class FP8GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{what}: " if what else ""
        super().__init__(f"{msg}{STATUS.get(status, status)} ({_status_string(status)})")


class _COptions(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("force_realign", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("stages", ctypes.c_int), ("splits", ctypes.c_int),
                ("no_workspace", ctypes.c_int), ("mma_ctas", ctypes.c_int),
                ("split_tail", ctypes.c_int), ("reserved", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("ldx", ctypes.c_size_t), ("ldw", ctypes.c_size_t),
                ("epilogue_warps", ctypes.c_int)]


_PLAN_INT_FIELDS = ("path", "realign", "tile_m", "tile_n", "stages", "splits", "grid", "cluster",
                    "threads", "smem_bytes", "launches", "repitch", "occupancy", "split_tiles",
                    "tail_workers")


class _CPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in _PLAN_INT_FIELDS] + [
        ("workspace_bytes", ctypes.c_size_t), ("epilogue_warps", ctypes.c_int),
        ("kblocks_per_stage", ctypes.c_int)]


@dataclass
class Options:
    path: int = PATH_AUTO
    force_realign: bool = False
    tile_n: int = 0
    stages: int = 0
    splits: int = 0
    no_workspace: bool = False
    mma_ctas: int = 0           # main path: 0 auto, 1 one-CTA tiles, 2 CTA-pair tiles
    split_tail: bool = False    # share the last partial wave's tiles out by K (needs a workspace)
    workspace: int = 0          # device pointer (e.g. tensor.data_ptr()), 0 = library pool
    workspace_bytes: int = 0
    ldx: int = 0                # row pitch of x in bytes, 0 = K (set from strided views)
    ldw: int = 0                # row pitch of w in bytes, 0 = K
    epilogue_warps: int = 0     # CTA-pair tiles: 0 auto, 4 or 8

    def _c(self) -> _COptions:
        o = _COptions()
        o.path, o.force_realign = int(self.path), int(bool(self.force_realign))
        o.tile_n, o.stages, o.splits = int(self.tile_n), int(self.stages), int(self.splits)
        o.no_workspace = int(bool(self.no_workspace))
        o.mma_ctas = int(self.mma_ctas)
        o.split_tail = int(bool(self.split_tail))
        o.workspace = int(self.workspace) or None
        o.workspace_bytes = int(self.workspace_bytes)
        o.ldx, o.ldw = int(self.ldx), int(self.ldw)
        o.epilogue_warps = int(self.epilogue_warps)
        return o


@dataclass
class Plan:
    path: int
    realign: int
    tile_m: int
    tile_n: int
    stages: int
    splits: int
    grid: int
    cluster: int
    threads: int
    smem_bytes: int
    launches: int
    repitch: int
    occupancy: int
    split_tiles: int
    tail_workers: int
    workspace_bytes: int
    epilogue_warps: int = 4
    kblocks_per_stage: int = 1


_lock = threading.RLock()
_lib = None


def library_path() -> Path:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _LIB_PATH.exists():
            raise FP8GemmError(3, f"CUDA library not built ({_LIB_PATH}); run "
                               "fp8_channel_scaled_gb300.build.build()")
        L = ctypes.CDLL(str(_LIB_PATH))
        vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        L.fp8_gemm_scaled.argtypes = [vp, vp, vp, vp, i, i, i, st]
        L.fp8_gemm_scaled_ex.argtypes = [vp, vp, vp, vp, i, i, i, ctypes.POINTER(_COptions), st]
        L.fp8_gemm_scaled_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, st]
        L.fp8_gemm_prepare_weight.argtypes = [vp, i, i, vp, ctypes.c_size_t, st]
        L.fp8_gemm_grouped.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(_COptions), st]
        L.fp8_gemm_plan.argtypes = [i, vp, vp, i, i, i, ctypes.POINTER(_COptions),
                                    ctypes.POINTER(_CPlan)]
        L.fp8_gemm_workspace_bytes.argtypes = [i, vp, vp, i, i, i, ctypes.POINTER(_COptions)]
        L.fp8_gemm_workspace_bytes.restype = ctypes.c_size_t
        L.fp8_gemm_check_device_error.argtypes = [st]
        L.fp8_gemm_set_wait_budget_ns.argtypes = [ctypes.c_ulonglong]
        L.fp8_gemm_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, st]
        L.fp8_gemm_status_string.argtypes = [i]
        L.fp8_gemm_status_string.restype = ctypes.c_char_p
        L.fp8_gemm_last_device_error_bits.argtypes = []
        L.fp8_gemm_last_device_error_bits.restype = ctypes.c_uint
        for f in ("fp8_gemm_scaled", "fp8_gemm_scaled_ex", "fp8_gemm_scaled_noalloc",
                  "fp8_gemm_prepare_weight", "fp8_gemm_grouped",
                  "fp8_gemm_plan",
                  "fp8_gemm_check_device_error", "fp8_gemm_set_wait_budget_ns",
                  "fp8_gemm_selftest_wait_timeout", "fp8_gemm_version"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
        return L


def _status_string(status: int) -> str:
    if _lib is None:
        return "library not loaded"
    return _lib.fp8_gemm_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    """Raw cudaStream_t of `stream` (None: the current device's current stream)."""
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:  # same value as current_stream().cuda_stream, without the object
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int:
    try:
        return t.data_ptr()
    except AttributeError:
        return int(t)


def _row_pitch(t, name):
    """Row pitch (elements) of a 2-D row-major view with unit inner stride."""
    if t.shape[0] <= 1 or t.is_contiguous():
        return int(t.shape[1])
    if t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must be row-major with unit inner stride")
    return int(t.stride(0))


def _shapes(x, w, scale, y, strided=False):
    xs, ws, ss, ys = x.shape, w.shape, scale.shape, y.shape
    if len(xs) != 2 or len(ws) != 2 or xs[1] != ws[1]:
        raise ValueError(f"x {tuple(xs)} and w {tuple(ws)} must be [M,K] and [N,K]")
    M, K = xs
    N = ws[0]
    if len(ss) != 1 or ss[0] != N or len(ys) != 2 or ys[0] != M or ys[1] != N:
        raise ValueError(f"scale {tuple(ss)} / y {tuple(ys)} do not match M={M} N={N}")
    if strided:
        if not x.is_contiguous():
            _row_pitch(x, "x")
        if not w.is_contiguous():
            _row_pitch(w, "w")
    elif not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError(("x" if not x.is_contiguous() else "w") + " must be contiguous")
    if not scale.is_contiguous():
        raise ValueError("scale must be contiguous")
    if not y.is_contiguous():
        raise ValueError("y must be contiguous")
    if x.element_size() != 1 or w.element_size() != 1:
        raise TypeError("x and w must be 1-byte E4M3 tensors (uint8 or float8_e4m3fn)")
    if scale.element_size() != 4 or y.element_size() != 2:
        raise TypeError("scale must be float32 and y bfloat16")
    return M, N, K


def _check(status: int, what: str):
    if status != 0:
        raise FP8GemmError(status, what)


# ---------------------------------------------------------------- same names as the C ABI
def fp8_gemm_scaled(x, w, scale, y, stream=None) -> None:
    """y = bf16((x . w^T, fp32 acc) * scale) on `stream` (torch tensors on one GPU)."""
    M, N, K = _shapes(x, w, scale, y)
    _check(lib().fp8_gemm_scaled(_ptr(x), _ptr(w), _ptr(scale), _ptr(y), M, N, K,
                                 _stream_handle(stream)), "fp8_gemm_scaled")


def fp8_gemm_scaled_ex(x, w, scale, y, options: Options | None = None, stream=None) -> None:
    """As fp8_gemm_scaled with options; x and w may be row-major views with a
    row pitch (e.g. buf[:, :K]): their pitches go to options.ldx / ldw."""
    M, N, K = _shapes(x, w, scale, y, strided=True)
    o = options._c() if options is not None else _COptions()  # all-zero: the defaults
    if not o.ldx and _row_pitch(x, "x") != K:
        o.ldx = _row_pitch(x, "x")
    if not o.ldw and _row_pitch(w, "w") != K:
        o.ldw = _row_pitch(w, "w")
    _check(lib().fp8_gemm_scaled_ex(_ptr(x), _ptr(w), _ptr(scale), _ptr(y), M, N, K,
                                    ctypes.byref(o), _stream_handle(stream)),
           "fp8_gemm_scaled_ex")


def fp8_gemm_scaled_noalloc(x, w, scale, y, stream=None) -> None:
    """As fp8_gemm_scaled, but allocates no device memory: any repitch copies go
    into the library's static 32 MiB device workspace (see include/fp8_gemm.h).
    Calls that overlap on the GPU race on that workspace."""
    M, N, K = _shapes(x, w, scale, y)
    _check(lib().fp8_gemm_scaled_noalloc(_ptr(x), _ptr(w), _ptr(scale), _ptr(y), M, N, K,
                                         _stream_handle(stream)), "fp8_gemm_scaled_noalloc")


def fp8_gemm_grouped(x, w, scale, y, offsets, options: Options | None = None, stream=None) -> None:
    """Grouped layer: x [M, K], w [G, N, K], scale [G, N], y [M, N], offsets
    int32 [G + 1] on the device (group g owns rows offsets[g] .. offsets[g+1])."""
    if x.dim() != 2 or w.dim() != 3 or scale.dim() != 2 or y.dim() != 2 or offsets.dim() != 1:
        raise ValueError("x [M,K], w [G,N,K], scale [G,N], y [M,N], offsets [G+1] expected")
    M, K = x.shape
    G, N, Kw = w.shape
    if Kw != K or tuple(scale.shape) != (G, N) or tuple(y.shape) != (M, N) or offsets.shape[0] != G + 1:
        raise ValueError("shapes do not match")
    for name, t in (("w", w), ("scale", scale), ("y", y), ("offsets", offsets)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if x.element_size() != 1 or w.element_size() != 1 or scale.element_size() != 4 \
            or y.element_size() != 2 or offsets.element_size() != 4:
        raise TypeError("x, w: 1-byte E4M3; scale: float32; y: bfloat16; offsets: int32")
    o = (options or Options())._c()
    if not o.ldx and _row_pitch(x, "x") != K:
        o.ldx = _row_pitch(x, "x")
    _check(lib().fp8_gemm_grouped(_ptr(x), _ptr(w), _ptr(scale), _ptr(y), _ptr(offsets), int(G),
                                  int(M), int(N), int(K), ctypes.byref(o), _stream_handle(stream)),
           "fp8_gemm_grouped")


def fp8_gemm_prepare_weight(w, w_out, stream=None):
    """Copy w [N, K] (contiguous) into the rows of w_out, a uint8 [N, ldw]
    buffer (ldw a multiple of 16, >= K; a multiple of 64 reads fastest),
    zeroing bytes past K; returns the [N, K] view of w_out to pass as w (its
    pitch reaches the library)."""
    if w.dim() != 2 or not w.is_contiguous() or w.element_size() != 1:
        raise ValueError("w must be a contiguous 2-D 1-byte tensor")
    N, K = w.shape
    if w_out.dim() != 2 or w_out.shape[0] != N or w_out.shape[1] < K or not w_out.is_contiguous():
        raise ValueError(f"w_out must be a contiguous [{N}, >= {K}] buffer")
    _check(lib().fp8_gemm_prepare_weight(_ptr(w), int(N), int(K), _ptr(w_out),
                                         int(w_out.shape[1]), _stream_handle(stream)),
           "fp8_gemm_prepare_weight")
    return w_out[:, :K]


def fp8_gemm_plan(device: int, M: int, N: int, K: int, options: Options | None = None,
                  x_ptr: int = 0, w_ptr: int = 0) -> Plan:
    o = (options or Options())._c()
    p = _CPlan()
    _check(lib().fp8_gemm_plan(int(device), x_ptr or None, w_ptr or None, int(M), int(N), int(K),
                               ctypes.byref(o), ctypes.byref(p)), "fp8_gemm_plan")
    return Plan(*[getattr(p, f) for f in _PLAN_INT_FIELDS], int(p.workspace_bytes),
                int(p.epilogue_warps), int(p.kblocks_per_stage))


def fp8_gemm_workspace_bytes(device: int, M: int, N: int, K: int, options: Options | None = None,
                             x_ptr: int = 0, w_ptr: int = 0) -> int:
    o = (options or Options())._c()
    return int(lib().fp8_gemm_workspace_bytes(int(device), x_ptr or None, w_ptr or None, int(M),
                                              int(N), int(K), ctypes.byref(o)))


def fp8_gemm_check_device_error(stream=None) -> int:
    """Synchronise `stream`, read and clear the device error word; returns the status."""
    return int(lib().fp8_gemm_check_device_error(_stream_handle(stream)))


def fp8_gemm_set_wait_budget_ns(ns: int) -> None:
    _check(lib().fp8_gemm_set_wait_budget_ns(int(ns)), "fp8_gemm_set_wait_budget_ns")


def fp8_gemm_selftest_wait_timeout(budget_ns: int, stream=None) -> None:
    _check(lib().fp8_gemm_selftest_wait_timeout(int(budget_ns), _stream_handle(stream)),
           "fp8_gemm_selftest_wait_timeout")


def fp8_gemm_status_string(status: int) -> str:
    return _status_string(status)


def fp8_gemm_version() -> int:
    return int(lib().fp8_gemm_version())


# ---------------------------------------------------------------- conveniences
def check_device_error(stream=None) -> None:
    """Raise if a kernel launched since the last check gave up a bounded wait."""
    st = fp8_gemm_check_device_error(stream)
    if st != 0:
        bits = int(lib().fp8_gemm_last_device_error_bits())
        raise FP8GemmError(st, f"device error bits 0x{bits:x}")


def plan(M: int, N: int, K: int, options: Options | None = None, device: int | None = None,
         x=None, w=None) -> Plan:
    if device is None:
        import torch
        device = torch.cuda.current_device()
    o = options or Options()
    if x is not None and hasattr(x, "stride") and not o.ldx and _row_pitch(x, "x") != K:
        o = dataclasses.replace(o, ldx=_row_pitch(x, "x"))
    if w is not None and hasattr(w, "stride") and not o.ldw and _row_pitch(w, "w") != K:
        o = dataclasses.replace(o, ldw=_row_pitch(w, "w"))
    return fp8_gemm_plan(device, M, N, K, o, _ptr(x) if x is not None else 0,
                         _ptr(w) if w is not None else 0)


def linear(x, w, scale, out=None, options: Options | None = None, stream=None):
    """Allocate (or reuse `out`) and return y = bf16((x . w^T) * scale)."""
    import torch
    if out is None:
        out = torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device=x.device)
    if options is None:
        fp8_gemm_scaled(x, w, scale, out, stream)
    else:
        fp8_gemm_scaled_ex(x, w, scale, out, options, stream)
    return out
