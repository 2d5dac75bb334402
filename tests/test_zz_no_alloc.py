"""fp8_gemm_scaled_noalloc, the allocation-free entry point, against
fp8_gemm_scaled.

Some callers cannot allocate device memory: code running inside another
framework's or allocator's memory accounting, in a process whose device
memory is fixed up front, or on a path that must not synchronise the device
the way cudaMalloc / cudaFree can.  For them the library offers one entry
point that calls no allocating routine; when the operands have to be
repitched (rows not 16-byte aligned, here K = 4127) it uses a static 32 MiB
device array instead of a workspace pool.

The array keeps the previous call's contents, so the test makes two calls in
a row with different data and checks each against the CPU oracle and against
the ordinary entry point, within the parity tolerance of the other GPU tests
(bitwise against the ordinary entry point when both run the same kernels on
the same repitched bytes), and checks that the device's free memory does not
change across the calls.  It goes through the C ABI directly.  This file is
collected last so that a run stopping at the first failure has run every
other test first.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import compare, to_dev, y_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import fp8_channel_scaled_gb300 as fg  # noqa: E402

ESIZE = 7


def _call(fn, x, w, s, y):
    lib = fg.lib()
    st = getattr(lib, fn)(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                          ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                          x.shape[0], w.shape[0], x.shape[1],
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_channel_scaled_gb300 import build
    build.build()
    fg.lib()


def _noalloc_plan(M, N, K):
    """What the no-alloc entry runs: the automatic plan with a caller workspace
    (which is what the static array is)."""
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    return fg.plan(M, N, K, options=fg.Options(workspace=ws.data_ptr(),
                                               workspace_bytes=fg.NOALLOC_WORKSPACE_BYTES))


def test_noalloc_matches_oracle_and_scaled_on_two_calls_in_a_row():
    M, N, K = 320, 528, 4127
    p = _noalloc_plan(M, N, K)
    assert p.repitch == 1  # the static workspace is really used
    assert p.workspace_bytes <= fg.NOALLOC_WORKSPACE_BYTES
    same_kernels = fg.plan(M, N, K) == p
    inputs = [synth.make_inputs(M, N, K, seed) for seed in (11, 12)]
    dev = [tuple(to_dev(a) for a in xws) for xws in inputs]
    y_na = [torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda") for _ in dev]
    y_ref = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in dev]
    for (xd, wd, sd), yr in zip(dev, y_ref):  # also loads every kernel module once
        assert _call("fp8_gemm_scaled", xd, wd, sd, yr) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for (xd, wd, sd), yn in zip(dev, y_na):
        assert _call("fp8_gemm_scaled_noalloc", xd, wd, sd, yn) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0  # nothing was allocated
    assert fg.fp8_gemm_check_device_error() == 0
    for seed, (x, w, s), yn, yr in zip((11, 12), inputs, y_na, y_ref):
        got = y_bits(yn)
        compare(got, oracle.linear(x, w, s), f"noalloc seed {seed} vs oracle")
        compare(got, y_bits(yr), f"noalloc seed {seed} vs fp8_gemm_scaled")
        if same_kernels:
            assert np.array_equal(got, y_bits(yr))


def test_noalloc_aligned_operands_and_size_limit():
    # aligned operands need no workspace: same kernels as the ordinary entry
    x, w, s = synth.make_inputs(256, 384, 1024, 13)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y_na = torch.empty((256, 384), dtype=torch.bfloat16, device="cuda")
    y_ref = torch.empty_like(y_na)
    assert _call("fp8_gemm_scaled_noalloc", xd, wd, sd, y_na) == 0
    assert _call("fp8_gemm_scaled", xd, wd, sd, y_ref) == 0
    assert fg.fp8_gemm_check_device_error() == 0
    compare(y_bits(y_na), y_bits(y_ref), "noalloc aligned")
    # a repitch that does not fit in the static array is refused, nothing runs
    M, N, K = 4096, 4096, 4127
    assert fg.plan(M, N, K).workspace_bytes > fg.NOALLOC_WORKSPACE_BYTES
    xb = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    wb = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sb = torch.ones(N, dtype=torch.float32, device="cuda")
    yb = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    assert _call("fp8_gemm_scaled_noalloc", xb, wb, sb, yb) == ESIZE
    assert fg.fp8_gemm_check_device_error() == 0
    assert bool(torch.all(yb == 5.0))
