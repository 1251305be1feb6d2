"""Pins for the fp64 oracle: what the pages and the mathematics fix, checked
against the oracle without any GPU.

Each test names the property it pins and where it comes from. Together they
are chosen so that a plausible slip in the oracle (a dropped eps, eps outside
the root, dividing by the padded width, a wrong index or stride, offset
multiplied instead of added, a double rounding, a wrong sign) fails at least
one of them.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from exact import decode_exact, round_exact, rmsnorm_row_exact
from memory_bound_normalization_fwd_gb300 import workloads as W

ALL = np.arange(65536, dtype=np.uint16)
F32 = np.float32


def _bits_of(dtype, values):
    """Exact small-format values -> bit patterns via the exact rounder (values are representable)."""
    return np.array([round_exact(dtype, Fraction(v)) for v in values], dtype=np.uint16)


def _rand_bits(rng, shape, dtype, scale=1.0):
    t = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
    return W.from_torch(t.to(torch.bfloat16 if dtype == "bf16" else torch.float16))


# ---------------------------------------------------------------- decoders

def test_decode_bf16_all_patterns_match_torch():
    ref = torch.from_numpy(ALL.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode("bf16", ALL)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_decode_fp16_all_patterns_match_numpy():
    ref = ALL.view(np.float16).astype(np.float64)
    got = oracle.decode("fp16", ALL)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


# ---------------------------------------------------------------- encoders

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_round_trips_every_pattern(dtype):
    vals = oracle.decode(dtype, ALL)
    finite = ~np.isnan(vals)
    assert np.array_equal(oracle.encode(dtype, vals[finite]), ALL[finite])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_midpoints_tie_to_even(dtype):
    # Every pair of neighbouring positive finite values: the exact midpoint goes
    # to the even pattern, one double above it to the upper, one below to the lower.
    inf_bits = 0x7F80 if dtype == "bf16" else 0x7C00
    lo_bits = np.arange(0, inf_bits - 1, dtype=np.uint16)
    hi_bits = lo_bits + 1
    lo = oracle.decode(dtype, lo_bits)
    hi = oracle.decode(dtype, hi_bits)
    mid = (lo + hi) / 2  # exact in fp64 (few significant bits)
    even = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(oracle.encode(dtype, mid), even)
    assert np.array_equal(oracle.encode(dtype, np.nextafter(mid, np.inf)), hi_bits)
    assert np.array_equal(oracle.encode(dtype, np.nextafter(mid, -np.inf)), lo_bits)
    assert np.array_equal(oracle.encode(dtype, -mid), even | 0x8000)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_overflow_threshold(dtype):
    mbits = 7 if dtype == "bf16" else 10
    inf_bits = 0x7F80 if dtype == "bf16" else 0x7C00
    max_bits = inf_bits - 1
    vmax = float(decode_exact(dtype, max_bits))
    half_ulp = float(Fraction(2) ** (math.floor(math.log2(vmax)) - mbits - 1))
    # The largest finite value has an odd significand, so its upper midpoint rounds to inf.
    assert oracle.encode(dtype, np.array([vmax + half_ulp]))[0] == inf_bits
    assert oracle.encode(dtype, np.array([np.nextafter(vmax + half_ulp, 0)]))[0] == max_bits
    assert oracle.encode(dtype, np.array([np.inf, -np.inf])).tolist() == [inf_bits, inf_bits | 0x8000]
    nan = oracle.encode(dtype, np.array([np.nan]))[0]
    assert (nan & inf_bits) == inf_bits and (nan & ((1 << mbits) - 1)) != 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_random_doubles_match_exact_rounding(dtype):
    rng = np.random.default_rng(1234)
    lo, hi = (-140, 130) if dtype == "bf16" else (-30, 17)
    v = rng.uniform(1, 2, 4000) * np.exp2(rng.integers(lo, hi, 4000)) * rng.choice([-1, 1], 4000)
    got = oracle.encode(dtype, v)
    want = np.array([round_exact(dtype, Fraction(float(t))) for t in v], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_encode_fp16_matches_numpy_direct_conversion():
    # numpy converts float64 -> float16 with a single rounding (no float32 step).
    rng = np.random.default_rng(7)
    v = rng.standard_normal(1 << 20) * np.exp2(rng.integers(-26, 17, 1 << 20))
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode("fp16", v), ref)


def test_encode_bf16_matches_torch_on_float32_values():
    # For values exactly representable in float32, torch's float32 -> bf16 is one RNE step.
    rng = np.random.default_rng(8)
    f = rng.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    f = f[np.isfinite(f)]
    want = W.from_torch(torch.from_numpy(f).to(torch.bfloat16))
    assert np.array_equal(oracle.encode("bf16", f.astype(np.float64)), want)


# ---------------------------------------------------------------- forward

def _fixture_cases():
    path = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.txt")
    cases, cur = [], None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("["):
            cur = {"name": line.strip("[]")}
            cases.append(cur)
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        cur[k] = v
    return cases


def _tokens(s):
    out = []
    for tok in s.split():
        if "*" in tok:
            v, k = tok.split("*")
            out += [Fraction(v)] * int(k)
        else:
            out.append(Fraction(tok))
    return out


@pytest.mark.parametrize("case", _fixture_cases(), ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    dtype = case["dtype"]
    x, w = _tokens(case["x"]), _tokens(case["w"])
    eps, offset = float(Fraction(case["eps"])), float(Fraction(case["offset"]))
    rstd_exact = Fraction(case["rstd"])
    y_exact, y_rounded = _tokens(case["y_exact"]), _tokens(case["y_rounded"])
    # The fixture's hand rounding agrees with the exact rounder.
    assert [round_exact(dtype, v) for v in y_exact] == [round_exact(dtype, v) for v in y_rounded]
    xb, wb = _bits_of(dtype, x), _bits_of(dtype, w)
    assert [decode_exact(dtype, int(b)) for b in xb] == x  # inputs are representable
    y, rstd, y64 = oracle.rmsnorm_fwd(xb[None, :], wb, eps, offset, dtype, want_y64=True)
    assert rstd[0] == pytest.approx(float(rstd_exact), rel=1e-15)
    assert np.allclose(y64[0], [float(v) for v in y_exact], rtol=1e-15, atol=0)
    got = [decode_exact(dtype, int(b)) for b in y[0]]
    assert got == y_rounded


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("N", [1, 7, 512, 1000])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_constant_row_closed_form(dtype, N, eps, offset):
    # A row x_j = c gives r = 1/sqrt(c^2 + eps) and y_j = c r (offset + w_j).
    rng = np.random.default_rng(N)
    cs = [1.0, -0.5, 3.0, 2.0 ** -8, 256.0 if dtype == "fp16" else 1024.0]
    xb = _bits_of(dtype, [Fraction(c) for c in cs])
    x = np.repeat(xb[:, None], N, axis=1)
    wb = _rand_bits(rng, (N,), dtype, 0.5)
    y, rstd = oracle.rmsnorm_fwd(x, wb, eps, offset, dtype)
    e = Fraction(float(F32(eps)))
    for i, c in enumerate(cs):
        assert rstd[i] == pytest.approx(1.0 / math.sqrt(c * c + float(e)), rel=1e-15)
        r, ys = rmsnorm_row_exact([Fraction(c)] * N,
                                  [decode_exact(dtype, int(b)) for b in wb], e, Fraction(offset))
        assert y[i].tolist() == [round_exact(dtype, v, negative_zero=(c < 0)) if v == 0
                                 else round_exact(dtype, v) for v in ys]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("k", [-8, -1, 1, 4])
def test_power_of_two_scale_invariance(dtype, k):
    # eps = 0: y(2^k x) == y(x) bit for bit and rstd(2^k x) == rstd(x) / 2^k exactly,
    # because scaling by a power of two commutes with every correctly rounded step.
    rng = np.random.default_rng(100 + k)
    # magnitudes in [0.5, 2) keep every scaled value normal in both formats
    mag = rng.uniform(0.5, 2.0, (16, 300)) * rng.choice([-1.0, 1.0], (16, 300))
    x = W.from_torch(torch.from_numpy(mag).to(torch.bfloat16 if dtype == "bf16" else torch.float16))
    w = _rand_bits(rng, (300,), dtype)
    xs = W.from_torch(W.to_torch(x, dtype).to(torch.float64).mul(2.0 ** k)
                      .to(torch.bfloat16 if dtype == "bf16" else torch.float16))
    assert np.array_equal(oracle.decode(dtype, xs), oracle.decode(dtype, x) * 2.0 ** k)
    y0, r0 = oracle.rmsnorm_fwd(x, w, 0.0, 0.0, dtype)
    y1, r1 = oracle.rmsnorm_fwd(xs, w, 0.0, 0.0, dtype)
    assert np.array_equal(y0, y1)
    assert np.array_equal(r1, r0 / 2.0 ** k)


def test_padding_columns_do_not_enter_the_sum():
    # Zero columns appended to a row change only the divisor: the sum of squares
    # recovered from rstd is the same, and the mean uses each row's own N.
    rng = np.random.default_rng(5)
    x = _rand_bits(rng, (8, 1000), "bf16")
    w = _rand_bits(rng, (1024,), "bf16")
    xp = np.zeros((8, 1024), dtype=np.uint16)
    xp[:, :1000] = x
    eps = 1e-6
    e = float(F32(eps))
    _, r = oracle.rmsnorm_fwd(x, w[:1000], eps, 0.0, "bf16")
    yp, rp = oracle.rmsnorm_fwd(xp, w, eps, 0.0, "bf16")
    s = 1000 * (1.0 / r ** 2 - e)
    sp = 1024 * (1.0 / rp ** 2 - e)
    assert np.allclose(s, sp, rtol=1e-12)
    assert np.all(oracle.decode("bf16", yp[:, 1000:]) == 0)  # +0 or -0 (sign of w)
    s_direct = (oracle.decode("bf16", x) ** 2).sum(axis=1)
    assert np.allclose(s, s_direct, rtol=1e-12)


def test_rows_are_independent():
    # Changing one row changes that row's outputs only (a stride or index slip breaks this).
    rng = np.random.default_rng(6)
    x = _rand_bits(rng, (5, 37), "bf16")
    w = _rand_bits(rng, (37,), "bf16")
    y0, r0 = oracle.rmsnorm_fwd(x, w, 1e-6, 0.0, "bf16")
    x2 = x.copy()
    x2[2] = _rand_bits(rng, (37,), "bf16", 3.0)
    y1, r1 = oracle.rmsnorm_fwd(x2, w, 1e-6, 0.0, "bf16")
    keep = [0, 1, 3, 4]
    assert np.array_equal(y0[keep], y1[keep]) and np.array_equal(r0[keep], r1[keep])
    assert not np.array_equal(y0[2], y1[2])
    # and the row range form returns the same rows
    yr, rr = oracle.rmsnorm_fwd(x, w, 1e-6, 0.0, "bf16", rows=(1, 4))
    assert np.array_equal(yr, y0[1:4]) and np.array_equal(rr, r0[1:4])


def test_fp16_workload_needs_fp32_accumulation():
    # The 131072x4096 fp16 workload draws x ~ N(0, 64^2): single squares and every
    # row's sum exceed the largest fp16 (65504), yet rstd stays finite near 1/64.
    wl = W.WORKLOADS["rmsnorm_131072x4096_fp16"]
    small = W.Workload("fp16_slice", 64, wl.N, dtype="fp16", x_std=wl.x_std)
    x, w = W.generate(small)
    xv = oracle.decode("fp16", x)
    assert (np.abs(xv) > 256).sum() > 5   # 4-sigma values: x^2 alone overflows fp16
    assert (xv ** 2).sum(axis=1).min() > 100 * 65504
    y, r = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp16")
    assert np.all(np.isfinite(r)) and abs(r.mean() * 64 - 1) < 0.02
    assert np.all(np.isfinite(oracle.decode("fp16", y)))


@pytest.mark.parametrize("offset", [0.0, 1.0])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_textbook_expression_in_torch_float64(offset, dtype):
    # The correctness reference the skillmd page gives,
    # x * rsqrt(mean(x^2) + eps) * weight, evaluated by torch in float64 with
    # weight = offset + w, matches the oracle's unrounded output.
    rng = np.random.default_rng(9)
    x = _rand_bits(rng, (32, 777), dtype, 2.0)
    w = _rand_bits(rng, (777,), dtype, 0.3)
    eps = 1e-5
    _, r, y64 = oracle.rmsnorm_fwd(x, w, eps, offset, dtype, want_y64=True)
    xt = W.to_torch(x, dtype).to(torch.float64)
    weight = offset + W.to_torch(w, dtype).to(torch.float64)
    e = float(F32(eps))
    rt = torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + e)
    ref = (xt * rt * weight).numpy()
    assert np.allclose(r, rt[:, 0].numpy(), rtol=1e-14, atol=0)
    assert np.allclose(y64, ref, rtol=1e-13, atol=1e-300)


def test_gemma_identity():
    # offset 1 with w = 0 is offset 0 with w = 1, bit for bit.
    rng = np.random.default_rng(10)
    x = _rand_bits(rng, (16, 513), "bf16")
    zeros = np.zeros(513, dtype=np.uint16)
    ones = _bits_of("bf16", [1] * 513)
    a = oracle.rmsnorm_fwd(x, zeros, 1e-6, 1.0, "bf16")
    b = oracle.rmsnorm_fwd(x, ones, 1e-6, 0.0, "bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_zero_row_eps_zero_gives_inf_and_nan():
    # A zero row with eps = 0: r = +inf and y = 0 * inf = NaN (IEEE).
    x = np.zeros((1, 4), dtype=np.uint16)
    w = _bits_of("bf16", [1] * 4)
    y, r = oracle.rmsnorm_fwd(x, w, 0.0, 0.0, "bf16")
    assert np.isinf(r[0]) and np.all(np.isnan(oracle.decode("bf16", y)))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_brute_force_tiny_shapes_against_exact_arithmetic(dtype):
    # Every M in 1..4 and N in 1..70 (fp16: a subset), random and integer inputs,
    # against exact rationals with a 60-digit square root.
    rng = np.random.default_rng(11 if dtype == "bf16" else 12)
    Ns = range(1, 71) if dtype == "bf16" else [1, 2, 3, 5, 8, 9, 16, 31, 33, 64, 70]
    for N in Ns:
        M = int(rng.integers(1, 5))
        if N % 3 == 0:
            x = _bits_of(dtype, [Fraction(int(v)) for v in rng.integers(-9, 10, M * N)]).reshape(M, N)
        else:
            x = _rand_bits(rng, (M, N), dtype, 1.5)
        w = _rand_bits(rng, (N,), dtype, 0.7)
        eps = float(rng.choice([0.0, 1e-6, 1e-5, 0.25]))
        offset = float(rng.choice([0.0, 1.0]))
        y, r = oracle.rmsnorm_fwd(x, w, eps, offset, dtype)
        wv = [decode_exact(dtype, int(b)) for b in w]
        for i in range(M):
            xv = [decode_exact(dtype, int(b)) for b in x[i]]
            rr, ys = rmsnorm_row_exact(xv, wv, Fraction(float(F32(eps))), Fraction(offset))
            if rr is None:   # all-zero row at eps = 0
                assert np.isinf(r[i])
                continue
            assert r[i] == pytest.approx(float(rr), rel=1e-15)
            for j, v in enumerate(ys):
                if v == 0:
                    assert decode_exact(dtype, int(y[i, j])) == 0
                else:
                    assert int(y[i, j]) == round_exact(dtype, v), (N, i, j)


def test_nan_and_inf_propagate_per_ieee():
    # A NaN in a row makes its sum, rstd and every y NaN; an Inf makes the sum
    # Inf and rstd 0, so y = x * 0 * s: +-0 everywhere except NaN at the Inf.
    x = _bits_of("bf16", [1, -2, 3, 4] * 3).reshape(3, 4)
    nan_b = np.uint16(0x7FC0)
    inf_b = np.uint16(0x7F80)
    x[1, 2] = nan_b
    x[2, 0] = inf_b
    w = _bits_of("bf16", [1, 1, 1, 1])
    y, r = oracle.rmsnorm_fwd(x, w, 1e-6, 0.0, "bf16")
    yv = oracle.decode("bf16", y)
    assert np.isfinite(r[0]) and np.all(np.isfinite(yv[0]))
    assert np.isnan(r[1]) and np.all(np.isnan(yv[1]))
    assert r[2] == 0.0 and np.isnan(yv[2, 0]) and np.all(yv[2, 1:] == 0)


def test_eps_is_taken_as_float32():
    # eps crosses the C boundary as fp32; the oracle must use exactly that value.
    x = _bits_of("bf16", [0, 0])
    w = _bits_of("bf16", [1, 1])
    _, r = oracle.rmsnorm_fwd(x[None, :], w, 1e-6, 0.0, "bf16")
    assert r[0] == 1.0 / math.sqrt(float(F32(1e-6)))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_single_rounding_just_below_a_tie(dtype):
    # x = (1, 1, 1, 1), eps = 2^-30 (exact in fp32), offset 1, w = 1.5 ulp(1):
    # y = (1 + 1.5 ulp) / sqrt(1 + 2^-30) lies about 2^-31 below the midpoint
    # between 1 + ulp (odd significand) and 1 + 2 ulp, so the one rounding the
    # pages' cast implies gives 1 + ulp. Rounding through fp32 first would land
    # exactly on the midpoint and round up to the even neighbour instead.
    ulp = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
    x = _bits_of(dtype, [1] * 4)[None, :]
    w = _bits_of(dtype, [Fraction(3, 2) * Fraction(ulp)] * 4)
    y, r, y64 = oracle.rmsnorm_fwd(x, w, 2.0 ** -30, 1.0, dtype, want_y64=True)
    mid = 1 + 1.5 * ulp
    assert y64[0, 0] < mid and mid - y64[0, 0] < 2.0 ** -30
    assert [decode_exact(dtype, int(b)) for b in y[0]] == [1 + Fraction(ulp)] * 4
