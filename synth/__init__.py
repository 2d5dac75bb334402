"""Seeded synthetic inputs for the scaled FP8 linear layer.

This module is shared by the tests, the smoke check and the benchmark.  It
draws the operands and quantises them to E4M3FN bytes; it holds none of the
layer's arithmetic (no decode, no dot product, no scaling, no bf16
rounding), and neither the CUDA library nor the oracle imports it.

Input recipe (the pages give no generator; this is the plainest reading of
the workload descriptions):

* ``rng = numpy.random.Generator(numpy.random.PCG64(seed))``
* draw order: ``x = rng.standard_normal((M, K))``, then
  ``w = rng.standard_normal((N, K))``, then ``u = rng.uniform(0.5, 1.5, N)``;
* ``weight_scale = (u / sqrt(K)).astype(float32)`` with the true K;
* outlier workloads only: ``n = round(0.01 * M * K)`` distinct flat positions
  ``rng.choice(M*K, n, replace=False)`` of x are replaced by
  ``448 * rng.choice([-1, 1], n)`` before quantisation;
* quantisation: E4M3FN, round to nearest even, directly from float64,
  saturating to +-448 (so no NaN is ever produced from a finite draw).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

E4M3_MAX = 448.0


def _e4m3_positive_values() -> np.ndarray:
    """The 127 non-negative finite E4M3FN values, index = code (0x00..0x7E)."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        vals[code] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_POS = _e4m3_positive_values()


def quantize_e4m3(v: np.ndarray) -> np.ndarray:
    """Encode float64 values as E4M3FN bytes: RNE, saturating to +-448.

    NaN encodes to 0x7F.  -0.0 keeps its sign (0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    # quantum of the binade a falls in: 2^(E-1-3) for normals, 2^-9 below 2^-6
    _, ex = np.frexp(a)                     # a = f * 2^ex, f in [0.5, 1)
    qexp = np.maximum(ex.astype(np.int32) - 4, -9).astype(np.int32)
    r = np.rint(np.ldexp(a, -qexp))         # rint: round half to even
    q = np.ldexp(r, qexp)                   # exact E4M3 magnitude (<= 448)
    code = np.searchsorted(_POS, q).astype(np.uint8)
    code = np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    outliers: bool = False

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Each operand read once, y written once: MK + NK + 4N + 2MN."""
        return self.M * self.K + self.N * self.K + 4 * self.N + 2 * self.M * self.N


WORKLOADS = {
    "small": Workload("small M=64,N=128,K=256", 64, 128, 256, 0),
    "square": Workload("square prefill M=N=K=4096", 4096, 4096, 4096, 1),
    "decode": Workload("decode M=32,N=8192,K=8192", 32, 8192, 8192, 2),
    "oddk": Workload("off-alignment K M=2048,N=4096,K=4127", 2048, 4096, 4127, 3),
    "mlp": Workload("MLP up-projection M=8192,N=14336,K=4096, 1% +-448 outliers",
                    8192, 14336, 4096, 4, outliers=True),
}


def make_inputs(M: int, N: int, K: int, seed: int, outliers: bool = False):
    """Return (x uint8 [M,K], w uint8 [N,K], weight_scale float32 [N])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    xf = rng.standard_normal((M, K))
    wf = rng.standard_normal((N, K))
    u = rng.uniform(0.5, 1.5, N)
    scale = (u / math.sqrt(K)).astype(np.float32)
    if outliers:
        n_out = int(round(0.01 * M * K))
        pos = rng.choice(M * K, n_out, replace=False)
        sgn = rng.choice(np.array([-1.0, 1.0]), n_out)
        xf.reshape(-1)[pos] = E4M3_MAX * sgn
    return quantize_e4m3(xf), quantize_e4m3(wf), scale


def workload_inputs(key: str):
    wl = WORKLOADS[key]
    return make_inputs(wl.M, wl.N, wl.K, wl.seed, wl.outliers)


def check_set(M: int, N: int, seed: int, n_rows: int = 64, n_elems: int = 8192):
    """Rows and elements checked on workloads too large for a full oracle pass.

    A separate stream (PCG64([seed, 1])) so the operand draws are unchanged:
    rows 0 and M-1 plus n_rows-2 distinct random rows, and n_elems (row, col)
    pairs drawn uniformly with replacement.
    """
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    n_rows = min(n_rows, M)
    fixed = np.unique(np.array([0, M - 1], dtype=np.int64))
    pool = np.setdiff1d(np.arange(M, dtype=np.int64), fixed)
    extra = rng.choice(pool, max(0, n_rows - fixed.size), replace=False) if pool.size else pool
    rows = np.sort(np.concatenate([fixed, np.asarray(extra, dtype=np.int64)]))[:n_rows]
    er = rng.integers(0, M, n_elems, dtype=np.int64)
    ec = rng.integers(0, N, n_elems, dtype=np.int64)
    return rows, er, ec
