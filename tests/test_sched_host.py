"""Host build of the tile scheduler (csrc/sched.cuh) checked on the CPU.

tests/sched_check.cpp includes the header with the CUDA qualifiers defined
away and checks, over thousands of seeded parameter sets: the grouped raster
visits every tile once; the split tail covers every (tile, K block) once, with
one owner per tile starting at K block 0, at most one published partial sum
per worker (its first tail unit), contributors owner+1 .. q_end-1 holding the
rest of the tile in order, a split tile as its owner's last unit, and at most
three segments per tile under the planner's worker count; the grouped-layer
mapper covers every row block and N block of every group once, inside the
group's clamped row range.
"""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def test_scheduler_invariants(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "sched_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-Wall", "-Werror",
                    "-I", str(ROOT / "fp8_channel_scaled_gb300" / "csrc"),
                    str(ROOT / "tests" / "sched_check.cpp"), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok "), r.stdout
