"""Parity on the five full-size workloads, in the launch configuration the
benchmark times (automatic path selection).

The decode and off-alignment-K workloads are checked on every output; the
square prefill and MLP up-projection workloads on 64 full rows (rows 0 and
M-1 among them) plus 8192 seeded random elements, which the oracle computes
one by one.
"""
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

FULL = {"small", "decode", "oddk"}


@pytest.mark.parametrize("key", ["small", "square", "decode", "oddk", "mlp"])
def test_workload(key):
    from fp8_channel_scaled_gb300 import build
    build.build()
    wl = synth.WORKLOADS[key]
    x, w, s = synth.workload_inputs(key)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
    p = fg.plan(wl.M, wl.N, wl.K, x=xd, w=wd)
    assert p.path == (fg.PATH_DECODE if wl.M <= 64 else fg.PATH_MAIN)
    odd = wl.K % 16 != 0
    assert p.repitch == int(odd) and p.realign == 0
    assert p.launches == (2 if odd else 1)
    fg.fp8_gemm_scaled(xd, wd, sd, y)
    fg.check_device_error()
    got = y_bits(y)
    if key in FULL:
        summary = compare(got, oracle.linear(x, w, s), key)
    else:
        rows, er, ec = synth.check_set(wl.M, wl.N, wl.seed)
        compare(got[rows], oracle.linear_rows(x, w, s, rows), f"{key} rows")
        summary = compare(got[er, ec], oracle.linear_elems(x, w, s, er, ec), f"{key} elements")
    # a second call into the same buffers must give the same bits
    fg.fp8_gemm_scaled(xd, wd, sd, y)
    fg.check_device_error()
    assert np.array_equal(y_bits(y), got)
    print(key, summary)
