"""Shared helpers for the GPU parity tests (no arithmetic of the layer)."""
from __future__ import annotations

import numpy as np

# Tolerance of the layer's output against the oracle, per element:
#   |y - y_ref| <= 2^-7 * |y_ref| + 1e-3
# (the workload's stated bound: one bf16 rounding is at most 2^-8 relative,
# fp32 accumulation of K <= 8192 products adds far less than another 2^-8).
REL_TOL = 2.0 ** -7
ABS_TOL = 1e-3


def bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def y_bits(y_torch) -> np.ndarray:
    """bf16 CUDA/CPU tensor -> numpy uint16 bit patterns."""
    import torch
    return y_torch.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compare(got_bits, ref_bits, what: str = "") -> dict:
    """Elementwise check within the tolerance; returns a summary, raises on a miss."""
    g = bits_to_f64(got_bits)
    r = bits_to_f64(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN pattern differs ({nan_g.sum()} vs {nan_r.sum()})"
    ok = ~nan_r
    err = np.abs(g[ok] - r[ok])
    bound = REL_TOL * np.abs(r[ok]) + ABS_TOL
    bad = err > bound
    summary = {
        "n": int(ok.sum()),
        "bad": int(bad.sum()),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_ratio": float((err / bound).max()) if err.size else 0.0,
        "bit_exact": float(np.mean(np.asarray(got_bits)[ok] == np.asarray(ref_bits)[ok])) if err.size else 1.0,
    }
    if summary["bad"]:
        idx = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {summary['bad']} of {summary['n']} outside tolerance; "
                             f"first {[(float(g[ok][i]), float(r[ok][i])) for i in idx]}; {summary}")
    return summary


def to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)
