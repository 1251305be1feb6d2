"""Pins for the oracle's fp32 activations (x, w and y in IEEE binary32).

The kernel listing of "Why cutile's rmsnorm required full register" (TileGym
issue #169) casts y back to the dtype of X, whatever it is; fp32 activations
take the same definition with binary32 as that dtype. These tests tie the
oracle's binary32 decoder and round-to-nearest-even encoder to numpy's float32
conversions (hardware IEEE conversions, a library independent of the oracle)
and to exact rational rounding, and its fp32 forward and backward to closed
forms, exact arithmetic and torch float64.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from exact import decode_exact, rmsnorm_row_exact, round_exact
from memory_bound_normalization_fwd_gb300 import workloads as W

F32 = np.float32
INF_BITS = 0x7F800000
MAX_BITS = 0x7F7FFFFF


def _sample_patterns() -> np.ndarray:
    """Every exponent with the extreme and a few random fractions, every
    subnormal near both ends of the range, and 2^20 random patterns."""
    rng = np.random.default_rng(21)
    expo = np.arange(256, dtype=np.uint32) << 23
    fracs = np.concatenate([np.array([0, 1, 2, 0x400000, 0x7FFFFE, 0x7FFFFF], dtype=np.uint32),
                            rng.integers(0, 1 << 23, 16, dtype=np.uint64).astype(np.uint32)])
    grid = (expo[:, None] | fracs[None, :]).ravel()
    sub = np.concatenate([np.arange(0, 1 << 16, dtype=np.uint32),
                          np.arange((1 << 23) - (1 << 16), 1 << 23, dtype=np.uint32)])
    rand = rng.integers(0, 1 << 32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    pos = np.concatenate([grid, sub, rand & 0x7FFFFFFF])
    return np.unique(np.concatenate([pos, pos | 0x80000000]))


PATTERNS = _sample_patterns()


def _bits_of(values) -> np.ndarray:
    return np.array([round_exact("fp32", Fraction(v)) for v in values], dtype=np.uint32)


def _rand(rng, shape, scale=1.0) -> np.ndarray:
    return (rng.standard_normal(shape) * scale).astype(np.float32).view(np.uint32)


# ---------------------------------------------------------------- decoder / encoder

def test_decode_matches_numpy_float32():
    with np.errstate(invalid="ignore"):  # signalling NaN patterns raise the flag when widened
        ref = PATTERNS.view(np.float32).astype(np.float64)
    got = oracle.decode("fp32", PATTERNS)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_decode_matches_exact_rationals_on_the_grid():
    for b in PATTERNS[:: max(1, PATTERNS.size // 3000)]:
        v = decode_exact("fp32", int(b))
        got = oracle.decode("fp32", np.array([b], dtype=np.uint32))[0]
        if v is None:
            assert not np.isfinite(got)
        else:
            assert Fraction(float(got)) == v


def test_encode_round_trips_sampled_patterns():
    vals = oracle.decode("fp32", PATTERNS)
    finite = ~np.isnan(vals)
    assert np.array_equal(oracle.encode("fp32", vals[finite]), PATTERNS[finite])


def test_encode_matches_numpy_float64_to_float32():
    # numpy's float64 -> float32 cast is one IEEE round-to-nearest-even step.
    rng = np.random.default_rng(22)
    n = 1 << 20
    v = rng.uniform(1, 2, n) * np.exp2(rng.integers(-160, 130, n)) * rng.choice([-1, 1], n)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float32).view(np.uint32)
    assert np.array_equal(oracle.encode("fp32", v), ref)


def test_encode_midpoints_tie_to_even():
    rng = np.random.default_rng(23)
    lo_bits = np.unique(np.concatenate([
        rng.integers(0, MAX_BITS, 1 << 16, dtype=np.uint64).astype(np.uint32),
        np.arange(0, 64, dtype=np.uint32),                     # smallest subnormals
        np.arange(0x007FFFF0, 0x00800010, dtype=np.uint32),    # subnormal/normal boundary
        np.arange(MAX_BITS - 32, MAX_BITS, dtype=np.uint32)]))
    hi_bits = lo_bits + 1
    lo, hi = oracle.decode("fp32", lo_bits), oracle.decode("fp32", hi_bits)
    mid = (lo + hi) / 2  # exact: 25 significant bits
    even = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(oracle.encode("fp32", mid), even)
    assert np.array_equal(oracle.encode("fp32", np.nextafter(mid, np.inf)), hi_bits)
    assert np.array_equal(oracle.encode("fp32", np.nextafter(mid, -np.inf)), lo_bits)
    assert np.array_equal(oracle.encode("fp32", -mid), even | 0x80000000)


def test_encode_overflow_threshold_and_specials():
    vmax = float(decode_exact("fp32", MAX_BITS))
    half_ulp = 2.0 ** (127 - 24)
    assert oracle.encode("fp32", np.array([vmax + half_ulp]))[0] == INF_BITS
    assert oracle.encode("fp32", np.array([np.nextafter(vmax + half_ulp, 0)]))[0] == MAX_BITS
    assert oracle.encode("fp32", np.array([np.inf, -np.inf])).tolist() == [INF_BITS,
                                                                            INF_BITS | 0x80000000]
    nan = int(oracle.encode("fp32", np.array([np.nan]))[0])
    assert (nan & INF_BITS) == INF_BITS and (nan & 0x7FFFFF) != 0
    assert oracle.encode("fp32", np.array([0.0, -0.0])).tolist() == [0, 0x80000000]
    # below half the smallest subnormal: zero; just above: the smallest subnormal
    tiny = 2.0 ** -149
    assert oracle.encode("fp32", np.array([tiny / 2, np.nextafter(tiny / 2, 1)])).tolist() == [0, 1]


def test_encode_random_doubles_match_exact_rounding():
    rng = np.random.default_rng(24)
    v = rng.uniform(1, 2, 3000) * np.exp2(rng.integers(-155, 129, 3000)) * rng.choice([-1, 1], 3000)
    got = oracle.encode("fp32", v)
    want = np.array([round_exact("fp32", Fraction(float(t))) for t in v], dtype=np.uint32)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("N", [1, 7, 512, 1000])
@pytest.mark.parametrize("eps", [0.0, 1e-6])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_constant_row_closed_form(N, eps, offset):
    # c stays below 2^12 so that c^2 + eps keeps eps in fp64: at c = 2^20 it
    # would round to c^2, and y = (offset + w) lands exactly on an fp32 tie that
    # the exact value misses by 1e-19 relative (the oracle is fp64, not exact).
    rng = np.random.default_rng(N + 5)
    cs = [1.0, -0.5, 3.0, 2.0 ** -8, 2.0 ** 10]
    x = np.repeat(_bits_of(cs)[:, None], N, axis=1)
    w = _rand(rng, (N,), 0.5)
    y, rstd = oracle.rmsnorm_fwd(x, w, eps, offset, "fp32")
    e = Fraction(float(F32(eps)))
    wv = [decode_exact("fp32", int(b)) for b in w]
    for i, c in enumerate(cs):
        assert rstd[i] == pytest.approx(1.0 / math.sqrt(c * c + float(e)), rel=1e-15)
        _, ys = rmsnorm_row_exact([Fraction(c)] * N, wv, e, Fraction(offset))
        assert y[i].tolist() == [round_exact("fp32", v, negative_zero=(c < 0)) if v == 0
                                 else round_exact("fp32", v) for v in ys]


@pytest.mark.parametrize("k", [-8, -1, 1, 4])
def test_power_of_two_scale_invariance(k):
    rng = np.random.default_rng(40 + k)
    mag = (rng.uniform(0.5, 2.0, (16, 300)) * rng.choice([-1.0, 1.0], (16, 300))).astype(np.float32)
    x = mag.view(np.uint32)
    xs = (mag * F32(2.0 ** k)).view(np.uint32)
    w = _rand(rng, (300,))
    y0, r0 = oracle.rmsnorm_fwd(x, w, 0.0, 0.0, "fp32")
    y1, r1 = oracle.rmsnorm_fwd(xs, w, 0.0, 0.0, "fp32")
    assert np.array_equal(y0, y1)
    assert np.array_equal(r1, r0 / 2.0 ** k)


@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_textbook_expression_in_torch_float64(offset):
    rng = np.random.default_rng(25)
    x, w = _rand(rng, (32, 777), 2.0), _rand(rng, (777,), 0.3)
    eps = 1e-5
    y, r, y64 = oracle.rmsnorm_fwd(x, w, eps, offset, "fp32", want_y64=True)
    xt = torch.from_numpy(x.view(np.float32)).to(torch.float64)
    weight = offset + torch.from_numpy(w.view(np.float32)).to(torch.float64)
    rt = torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + float(F32(eps)))
    ref = xt * rt * weight
    assert np.allclose(r, rt[:, 0].numpy(), rtol=1e-14, atol=0)
    assert np.allclose(y64, ref.numpy(), rtol=1e-13, atol=1e-300)
    # and y is torch's own float64 -> float32 rounding of that value (to within
    # the fp64 evaluation-order difference, which moves no rounding here)
    assert np.array_equal(y, ref.to(torch.float32).numpy().view(np.uint32))


def test_brute_force_tiny_shapes_against_exact_arithmetic():
    rng = np.random.default_rng(26)
    for N in [1, 2, 3, 4, 5, 8, 9, 16, 31, 33, 64, 70]:
        M = int(rng.integers(1, 4))
        if N % 3 == 0:
            x = _bits_of([Fraction(int(v)) for v in rng.integers(-9, 10, M * N)]).reshape(M, N)
        else:
            x = _rand(rng, (M, N), 1.5)
        w = _rand(rng, (N,), 0.7)
        eps = float(rng.choice([0.0, 1e-6, 0.25]))
        offset = float(rng.choice([0.0, 1.0]))
        y, r = oracle.rmsnorm_fwd(x, w, eps, offset, "fp32")
        wv = [decode_exact("fp32", int(b)) for b in w]
        for i in range(M):
            xv = [decode_exact("fp32", int(b)) for b in x[i]]
            rr, ys = rmsnorm_row_exact(xv, wv, Fraction(float(F32(eps))), Fraction(offset))
            if rr is None:
                assert np.isinf(r[i])
                continue
            assert r[i] == pytest.approx(float(rr), rel=1e-15)
            for j, v in enumerate(ys):
                if v == 0:
                    assert decode_exact("fp32", int(y[i, j])) == 0
                else:
                    assert int(y[i, j]) == round_exact("fp32", v), (N, i, j)


def test_gemma_identity():
    rng = np.random.default_rng(27)
    x = _rand(rng, (16, 513))
    a = oracle.rmsnorm_fwd(x, np.zeros(513, dtype=np.uint32), 1e-6, 1.0, "fp32")
    b = oracle.rmsnorm_fwd(x, _bits_of([1] * 513), 1e-6, 0.0, "fp32")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_single_rounding_just_below_a_tie():
    # x = (1, 1, 1, 1), eps = 2^-30, offset 1, w = 1.5 ulp(1) = 3 * 2^-24: y lies
    # about 2^-31 below the midpoint between 1 + ulp (odd) and 1 + 2 ulp, so it
    # rounds down to 1 + ulp.
    ulp = Fraction(1, 1 << 23)
    x = _bits_of([1] * 4)[None, :]
    w = _bits_of([Fraction(3, 2) * ulp] * 4)
    y, _, y64 = oracle.rmsnorm_fwd(x, w, 2.0 ** -30, 1.0, "fp32", want_y64=True)
    mid = 1 + 1.5 * float(ulp)
    assert y64[0, 0] < mid and mid - y64[0, 0] < 2.0 ** -30
    assert [decode_exact("fp32", int(b)) for b in y[0]] == [1 + ulp] * 4


def test_workload_generator_keeps_the_fp32_draws():
    wl = W.custom(3, 40, "fp32", seed=4)
    x, w = W.generate(wl)
    assert x.dtype == np.uint32 and w.dtype == np.uint32
    g = torch.Generator(device="cpu")
    g.manual_seed(4)
    xt = torch.randn((3, 40), generator=g, dtype=torch.float32)
    assert np.array_equal(x, xt.numpy().view(np.uint32))
    assert wl.algorithmic_bytes == 4 * 3 * 40 * 2 + 4 * 40 + 4 * 3
    assert np.array_equal(W.from_torch(W.to_torch(x, "fp32")), x)


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("offset", [0.0, 1.0])
@pytest.mark.parametrize("N", [1, 64, 1000])
def test_backward_matches_torch_float64_autograd(offset, N):
    rng = np.random.default_rng(N + 50)
    M = 7
    x, dy, w = _rand(rng, (M, N), 2.0), _rand(rng, (M, N)), _rand(rng, (N,), 0.4)
    eps = 1e-5
    e = float(F32(eps))
    xt = torch.from_numpy(x.view(np.float32)).to(torch.float64).requires_grad_(True)
    wt = torch.from_numpy(w.view(np.float32)).to(torch.float64).requires_grad_(True)
    gt = torch.from_numpy(dy.view(np.float32)).to(torch.float64)
    y = xt * torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + e) * (offset + wt)
    (y * gt).sum().backward()
    dx, dx64, dw = oracle.rmsnorm_bwd(x, w, dy, offset, "fp32", eps=eps)
    with torch.no_grad():
        r = torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + e)
        terms = (r * gt.abs() * (offset + wt).abs()).numpy()
    assert np.all(np.abs(dx64 - xt.grad.numpy()) <= 1e-11 * np.abs(dx64) + 1e-13 * terms)
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-13 * np.abs(dw).max())
    assert np.array_equal(dx, oracle.encode("fp32", dx64))
