"""Pins for the CPU oracle, checked against things other than the oracle.

Each pin is chosen so that a plausible slip in the oracle (a wrong exponent
bias, a dropped subnormal case, a transposed operand, a missing scale,
double rounding, a wrong tie rule) fails at least one of them:

* the E4M3FN code table against the format's fixed points (golden file) and
  against two independent decoders (torch.float8_e4m3fn, ml_dtypes);
* bf16 rounding against exact rational arithmetic (fractions.Fraction),
  including constructed midpoints;
* whole-layer brute force on tiny inputs in exact rational arithmetic;
* the exact dot against numpy's fp64 matmul of independently decoded
  operands (exact for these sizes, so any correct summation agrees);
* closed forms: one-hot weights reproduce x, power-of-two scales scale y
  exactly, zero x gives zero y, row/column permutations commute, zero
  K padding leaves y unchanged.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3fn_spec_points.txt")


# ---------------------------------------------------------------- helpers
def frac_e4m3(code: int):
    """E4M3FN value as an exact Fraction, or None for NaN (bit fields)."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None
    v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -v if s else v


def frac_rne_bf16_bits(v: Fraction) -> int:
    """bf16 bits of the exact rational v rounded to nearest, ties to even."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** max(e - 7, -133)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    res = fl * q
    if res > Fraction(2 ** 8 - 1, 2 ** 7) * Fraction(2) ** 127:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(res)))[0]
    assert float(res) == res
    return sign | (bits >> 16)


def torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def bf16_bits_of_fp32(f: np.ndarray) -> np.ndarray:
    """bf16 bits of values known to be exactly representable in bf16."""
    b = np.asarray(f, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


# ---------------------------------------------------------------- e4m3 table
def test_e4m3_golden_spec_points():
    tab = oracle.e4m3_table()
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code_s, val_s = line.split()
            code = int(code_s, 16)
            if val_s == "nan":
                assert math.isnan(tab[code]), hex(code)
            else:
                v = float(val_s)
                assert tab[code] == v and math.copysign(1, tab[code]) == math.copysign(1, v), hex(code)
            n += 1
    assert n >= 16


def test_e4m3_table_vs_torch_all_codes():
    tab = oracle.e4m3_table()
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(tab[~nan], ref[~nan])
    assert np.array_equal(np.signbit(tab[~nan]), np.signbit(ref[~nan]))
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0
    assert np.isfinite(tab).sum() == 254


def test_e4m3_table_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    tab = oracle.e4m3_table()
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert np.array_equal(tab[~nan], ref[~nan])


def test_e4m3_table_vs_fraction_bitfields():
    tab = oracle.e4m3_table()
    for c in range(256):
        fv = frac_e4m3(c)
        if fv is None:
            assert math.isnan(tab[c])
        else:
            assert Fraction(tab[c]) == fv, hex(c)


# ---------------------------------------------------------------- input encoder
def test_quantize_matches_torch_on_float32_values():
    rng = np.random.default_rng(123)
    v = np.concatenate([
        rng.standard_normal(200000) * rng.choice([1e-3, 1e-2, 0.1, 1, 10, 100], 200000),
        rng.uniform(-447.9, 447.9, 50000),
    ]).astype(np.float32).astype(np.float64)
    # every midpoint between neighbouring finite codes (exactly float32)
    pos = np.sort(oracle.e4m3_table()[:127])
    mids = (pos[:-1] + pos[1:]) / 2
    v = np.concatenate([v, mids, -mids, pos, -pos])
    ours = synth.quantize_e4m3(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_quantize_saturates_and_nan():
    v = np.array([448.0, 464.0, 1e30, -470.0, -1e30, np.inf, -np.inf, np.nan])
    assert synth.quantize_e4m3(v).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7E, 0xFE, 0x7F]


def test_generator_is_deterministic_and_shaped():
    x1, w1, s1 = synth.make_inputs(8, 16, 40, 7)
    x2, w2, s2 = synth.make_inputs(8, 16, 40, 7)
    assert x1.shape == (8, 40) and w1.shape == (16, 40) and s1.shape == (16,)
    assert np.array_equal(x1, x2) and np.array_equal(w1, w2) and np.array_equal(s1, s2)
    assert s1.dtype == np.float32
    u = s1.astype(np.float64) * math.sqrt(40)
    assert np.all(u > 0.49) and np.all(u < 1.51)


def test_generator_outliers():
    x, _, _ = synth.make_inputs(64, 8, 100, 4, outliers=True)
    n448 = int(np.sum((x == 0x7E) | (x == 0xFE)))
    assert n448 >= 64  # 1% of 6400 = 64 planted; N(0,1) never reaches 448 by itself


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rounding_vs_fraction_random():
    rng = np.random.default_rng(5)
    for _ in range(4000):
        d = float(rng.integers(-(2 ** 40), 2 ** 40)) * 2.0 ** -18
        s = np.float32(rng.uniform(1e-3, 2.0) * (1 if rng.random() < 0.5 else -1))
        want = frac_rne_bf16_bits(Fraction(d) * Fraction(float(s)))
        assert oracle.bf16_of_product(d, float(s)) == want, (d, s)


def test_bf16_rounding_midpoints_use_the_exact_product():
    # d * s placed exactly on a bf16 midpoint, then nudged by the smallest
    # amount d can move (2^-18): the exact product decides the direction.
    cases = 0
    for mant in (0x80, 0x81, 0x82, 0xFE, 0xFF):
        for ex in (-3, 0, 4):
            mid = Fraction(2 * mant + 1, 2 ** 8) * Fraction(2) ** ex   # between mant/128 and (mant+1)/128
            for s in (1.0, 0.5, 3.0, 0.75):
                for nudge in (-1, 0, 1):
                    d = mid / Fraction(s) + nudge * Fraction(1, 2 ** 18)
                    if d.denominator > 2 ** 18 or (d * 2 ** 18).denominator != 1:
                        continue
                    exact = d * Fraction(s)
                    got = oracle.bf16_of_product(float(d), s)
                    assert got == frac_rne_bf16_bits(exact), (mant, ex, s, nudge)
                    cases += 1
    assert cases > 60


def test_bf16_rounding_tiny_product_error_breaks_tie():
    # fl64(d*s) lands exactly on a bf16 midpoint although d*s does not; a
    # double-rounding oracle would apply ties-to-even here and be wrong
    # about half the time.
    rng = np.random.default_rng(17)
    seen = {+1: 0, -1: 0}
    for _ in range(20000):
        s = float(np.float32(rng.uniform(0.5, 2.0)))
        mid = (257 + 2 * int(rng.integers(128))) / 256.0 * 2.0 ** int(rng.integers(-4, 4))
        d = mid / s
        if d * s != mid:
            continue
        err = Fraction(d) * Fraction(s) - Fraction(mid)
        if err == 0:
            continue
        seen[1 if err > 0 else -1] += 1
        exact = Fraction(d) * Fraction(s)
        assert oracle.bf16_of_product(d, s) == frac_rne_bf16_bits(exact), (d, s)
    assert seen[1] > 100 and seen[-1] > 100


# ---------------------------------------------------------------- whole layer
def brute_force_bits(x, w, scale):
    M, K = x.shape
    N = w.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    nan = np.zeros((M, N), dtype=bool)
    for m in range(M):
        for n in range(N):
            terms = [(frac_e4m3(int(x[m, k])), frac_e4m3(int(w[n, k]))) for k in range(K)]
            if any(a is None or b is None for a, b in terms):
                nan[m, n] = True
                continue
            acc = sum((a * b for a, b in terms), Fraction(0))
            out[m, n] = frac_rne_bf16_bits(acc * Fraction(float(scale[n])))
    return out, nan


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_4x4x8(seed):
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    x = rng.choice(finite, (4, 8)).astype(np.uint8)
    w = rng.choice(finite, (4, 8)).astype(np.uint8)
    scale = rng.uniform(0.01, 3.0, 4).astype(np.float32)
    want, nan = brute_force_bits(x, w, scale)
    got = oracle.linear(x, w, scale, nthreads=3)
    ok = ~nan
    # signed zeros: compare values, not bits, where the exact result is 0
    gz = oracle.bf16_bits_to_f64(got)
    wz = oracle.bf16_bits_to_f64(want)
    assert np.array_equal(gz[ok], wz[ok])
    nz = ok & (wz != 0)
    assert np.array_equal(got[nz], want[nz])


def test_brute_force_subnormal_heavy():
    rng = np.random.default_rng(99)
    sub = np.array(list(range(0, 8)) + list(range(0x80, 0x88)) + [0x08, 0x88, 0x7E, 0xFE], dtype=np.uint8)
    x = rng.choice(sub, (4, 8)).astype(np.uint8)
    w = rng.choice(sub, (4, 8)).astype(np.uint8)
    scale = np.array([1.0, 2.0 ** -20, 3.0, 0.1], dtype=np.float32)
    want, _ = brute_force_bits(x, w, scale)
    got = oracle.linear(x, w, scale)
    assert np.array_equal(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(want))


def test_nan_operand_propagates():
    x, w, s = synth.make_inputs(3, 5, 16, 1)
    x = x.copy()
    x[1, 7] = 0x7F
    y = oracle.bf16_bits_to_f64(oracle.linear(x, w, s))
    assert np.all(np.isnan(y[1])) and not np.any(np.isnan(y[[0, 2]]))


def test_dot_equals_numpy_fp64_matmul():
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    x = rng.choice(finite, (37, 300)).astype(np.uint8)
    w = rng.choice(finite, (53, 300)).astype(np.uint8)
    want = torch_decode(x) @ torch_decode(w).T
    assert np.array_equal(oracle.dot(x, w, nthreads=5), want)


def test_dot_exact_at_large_k_with_outliers():
    # products up to 448^2 summed over K=8192: still exact, any order
    rng = np.random.default_rng(11)
    x = rng.choice(np.array([0x7E, 0xFE, 0x01, 0x81, 0x38], np.uint8), (4, 8192)).astype(np.uint8)
    w = rng.choice(np.array([0x7E, 0xFE, 0x01, 0x81, 0x39], np.uint8), (6, 8192)).astype(np.uint8)
    xd, wd = torch_decode(x), torch_decode(w)
    exact = [[sum(Fraction(a) * Fraction(b) for a, b in zip(xd[i], wd[j])) for j in range(6)] for i in range(4)]
    got = oracle.dot(x, w)
    assert all(Fraction(got[i, j]) == exact[i][j] for i in range(4) for j in range(6))


def test_one_hot_weight_reproduces_x():
    x, _, _ = synth.make_inputs(16, 8, 24, 2)
    K = 24
    w = np.zeros((K, K), dtype=np.uint8)
    w[np.arange(K), np.arange(K)] = 0x38            # 1.0
    scale = np.ones(K, dtype=np.float32)
    y = oracle.linear(x, w, scale)
    ref = torch.from_numpy(x).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xv = torch_decode(x)
    nz = xv != 0
    assert np.array_equal(y[nz], ref[nz])
    assert np.all(oracle.bf16_bits_to_f64(y[~nz]) == 0)


def test_power_of_two_scale_is_exact():
    x, w, _ = synth.make_inputs(9, 11, 64, 6)
    s1 = np.ones(11, dtype=np.float32)
    y1 = oracle.bf16_bits_to_f64(oracle.linear(x, w, s1))
    for j in (-12, -3, 5):
        yj = oracle.bf16_bits_to_f64(oracle.linear(x, w, s1 * np.float32(2.0 ** j)))
        assert np.array_equal(yj, y1 * 2.0 ** j)


def test_scale_is_applied_per_output_channel_not_per_row():
    x, w, s = synth.make_inputs(5, 7, 32, 8)
    d = oracle.dot(x, w)
    y = oracle.linear(x, w, s)
    for m in range(5):
        for n in range(7):
            assert y[m, n] == frac_rne_bf16_bits(Fraction(d[m, n]) * Fraction(float(s[n])))


def test_zero_x_gives_zero_y():
    _, w, s = synth.make_inputs(4, 9, 40, 3)
    y = oracle.linear(np.zeros((4, 40), np.uint8), w, s)
    assert np.all(oracle.bf16_bits_to_f64(y) == 0)


def test_permutation_equivariance():
    x, w, s = synth.make_inputs(12, 10, 48, 9)
    y = oracle.linear(x, w, s)
    rng = np.random.default_rng(1)
    pm, pn = rng.permutation(12), rng.permutation(10)
    yp = oracle.linear(x[pm], w[pn], s[pn])
    assert np.array_equal(yp, y[pm][:, pn])
    # a shared permutation of K leaves y unchanged
    pk = rng.permutation(48)
    assert np.array_equal(oracle.linear(x[:, pk], w[:, pk], s), y)


def test_zero_k_padding_is_invariant():
    x, w, s = synth.make_inputs(16, 24, 4127 // 16, 10)
    K = x.shape[1]
    y = oracle.linear(x, w, s)
    for Kp in (K + 1, 4224):
        xp = np.zeros((16, Kp), np.uint8)
        wp = np.zeros((24, Kp), np.uint8)
        xp[:, :K] = x
        wp[:, :K] = w
        assert np.array_equal(oracle.linear(xp, wp, s), y)
    # negative zero bytes (0x80) are zeros too
    xp = np.full((16, K + 5), 0x80, np.uint8)
    xp[:, :K] = x
    wp = np.zeros((24, K + 5), np.uint8)
    wp[:, :K] = w
    assert np.array_equal(oracle.linear(xp, wp, s), y)


def test_rows_and_elems_agree_with_full_and_threads():
    x, w, s = synth.make_inputs(33, 17, 130, 12)
    y = oracle.linear(x, w, s, nthreads=1)
    assert np.array_equal(oracle.linear(x, w, s, nthreads=7), y)
    rows = np.array([32, 0, 5, 5])
    assert np.array_equal(oracle.linear_rows(x, w, s, rows), y[rows])
    r = np.array([0, 32, 7, 7, 19])
    c = np.array([16, 0, 3, 3, 9])
    assert np.array_equal(oracle.linear_elems(x, w, s, r, c), y[r, c])


def test_empty_shapes():
    y = oracle.linear(np.zeros((0, 8), np.uint8), np.zeros((3, 8), np.uint8), np.ones(3, np.float32))
    assert y.shape == (0, 3)
    y = oracle.linear(np.zeros((2, 0), np.uint8), np.zeros((3, 0), np.uint8), np.ones(3, np.float32))
    assert np.all(oracle.bf16_bits_to_f64(y) == 0)


def test_check_set_shape():
    rows, er, ec = synth.check_set(8192, 14336, 4)
    assert rows.size == 64 and rows[0] == 0 and rows[-1] == 8191 and np.unique(rows).size == 64
    assert er.size == ec.size == 8192 and er.max() < 8192 and ec.max() < 14336
