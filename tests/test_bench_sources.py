"""bench.py reports a kernel's recorded DRAM traffic only while that kernel's
sources hash to the recorded value, so each per-kernel source list must name
every local file the kernel is compiled from (its .cu and, transitively, the
headers it includes); a list that missed one would keep stale counters."""
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fp8_channel_scaled_gb300", "csrc")


def _local_includes(path, seen=None):
    seen = set() if seen is None else seen
    with open(path) as f:
        for name in re.findall(r'^#include "([^"]+)"', f.read(), re.M):
            if name in seen:
                continue
            seen.add(name)
            inc = os.path.join(CSRC, name)
            if os.path.exists(inc):
                _local_includes(inc, seen)
    return seen


def _closure(cu):
    return {cu} | _local_includes(os.path.join(CSRC, cu))


def _names(paths):
    return {os.path.basename(p) for p in paths}


def test_pair_kernel_sources_are_complete():
    assert _names(bench.TC2_SOURCES) == _closure("gemm_tc2.cu")


def test_one_cta_kernel_sources_are_complete():
    assert _names(bench.TC_SOURCES) == _closure("gemm_tc.cu")


def test_decode_kernel_sources_are_complete():
    assert _names(bench.DEC_SOURCES) == _closure("gemm_decode.cu")


def test_recorded_traffic_table_parses():
    # the table holds one row per timed workload kernel; a hash that no longer
    # matches the sources yields None, never a stale number
    for key, srcs in (("square", bench.TC2_SOURCES), ("decode", bench.DEC_SOURCES)):
        t = bench.recorded_traffic(key, srcs)
        assert t is None or t > 0
    assert bench.recorded_traffic("square", bench.DEC_SOURCES) is None
