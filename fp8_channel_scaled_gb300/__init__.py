"""GB300 (sm_103a) per-output-channel scaled FP8 linear layer.

    y[M, N] = bf16((x_e4m3[M, K] . w_e4m3[N, K]^T, fp32 accumulate) * weight_scale[N])

This package is a thin ctypes binding over the C ABI in ``include/fp8_gemm.h``
(``_lib/libfp8gemm.so``, built in-tree by ``build.py``).  Every step of the
computation runs in the library's CUDA kernels; PyTorch only supplies device
memory and streams.  There is no fallback: if the library is missing or the
device is not a compute-capability-10.3 GPU, calls raise.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    FP8GemmError,
    NOALLOC_WORKSPACE_BYTES,
    Options,
    Plan,
    PATH_AUTO,
    PATH_DECODE,
    PATH_MAIN,
    STATUS,
    check_device_error,
    fp8_gemm_check_device_error,
    fp8_gemm_grouped,
    fp8_gemm_plan,
    fp8_gemm_prepare_weight,
    fp8_gemm_scaled,
    fp8_gemm_scaled_ex,
    fp8_gemm_scaled_noalloc,
    fp8_gemm_selftest_wait_timeout,
    fp8_gemm_set_wait_budget_ns,
    fp8_gemm_status_string,
    fp8_gemm_version,
    fp8_gemm_workspace_bytes,
    lib,
    library_path,
    linear,
    plan,
)
