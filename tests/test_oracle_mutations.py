"""The oracle's pins are sensitive: each plausible slip, planted in a scratch
copy of the oracle's C source, compiled on the CPU, must fail them.

The mutants never touch the repository's oracle; they live in a temporary
directory for the length of the test.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from exact import decode_exact, rmsnorm_row_exact, round_exact

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "rmsnorm_oracle.c")

MUTATIONS = {
    "eps outside the root": ("double r = 1.0 / sqrt(ms + e);", "double r = 1.0 / sqrt(ms) + e;"),
    "eps dropped": ("double r = 1.0 / sqrt(ms + e);", "double r = 1.0 / sqrt(ms);"),
    "divides by the padded width": ("double ms = s / (double)N;",
                                    "double ms = s / (double)((N + 7) / 8 * 8);"),
    "offset multiplied": ("double scale = off + load_elem(dtype, w, j);",
                          "double scale = (off == 0.0 ? 1.0 : off) * load_elem(dtype, w, j);"),
    "weight indexed by row": ("double scale = off + load_elem(dtype, w, j);",
                              "double scale = off + load_elem(dtype, w, (i + j) % N);"),
    "double rounding through fp32": ("if (y) store_elem(dtype, y, i * N + j, v);",
                                     "if (y) store_elem(dtype, y, i * N + j, (double)(float)v);"),
    "ties rounded down": ("if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;",
                          "if (rem > 0.5) n += 1.0;"),
    "sign of x lost": ("double v = load_elem(dtype, x, xi + j) * r * scale;",
                       "double v = fabs(load_elem(dtype, x, xi + j)) * r * scale;"),
    "sum of |x| instead of x^2": ("s += v * v;", "s += fabs(v);"),
    "wrong row stride": ("const int64_t xi = i * N;",
                         "const int64_t xi = i * (N > 1 ? N - 1 : N);"),
    "subnormal quantum off by one": ("if (e < emin) e = emin;", "if (e < emin - 1) e = emin - 1;"),
    "mean over N+1": ("double ms = s / (double)N;", "double ms = s / (double)(N + 1);"),
    "fp32 exponent bias off by one": ("mag = ldexp((double)((1 << 23) + frac), expo - 127 - 23);",
                                      "mag = ldexp((double)((1 << 23) + frac), expo - 126 - 23);"),
    "fp32 subnormal scale": ("mag = ldexp((double)frac, -126 - 23);",
                             "mag = ldexp((double)frac, -127 - 23);"),
    "fp32 encoder fraction bits": ("return round_to_binary(v, 23, -126, 127, 0xFF, 31);",
                                   "return round_to_binary(v, 22, -126, 127, 0xFF, 31);"),
}


def _build(tmp, source: str) -> ctypes.CDLL:
    c = os.path.join(tmp, "m.c")
    so = os.path.join(tmp, f"m{abs(hash(source))}.so")
    with open(c, "w") as f:
        f.write(source)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", so,
                    c, "-lm"], check=True)
    L = ctypes.CDLL(so)
    vp, f64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
    L.oracle_rmsnorm_fwd.argtypes = [vp, vp, vp, f64p, f64p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_int64]
    L.oracle_rmsnorm_bwd.argtypes = [vp, vp, vp, f64p, vp, f64p, f64p, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_float, ctypes.c_float, ctypes.c_int]
    L.oracle_encode.argtypes = [ctypes.c_int, ctypes.c_int64, f64p, vp]
    L.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_int64, vp, f64p]
    return L


CODE = {"bf16": 0, "fp16": 1, "fp32": 2}
BITS = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.uint32}


def _fwd(L, x, w, eps, offset, dtype):
    x = np.ascontiguousarray(x, dtype=BITS[dtype])
    w = np.ascontiguousarray(w, dtype=BITS[dtype])
    M, N = x.shape
    y = np.zeros((M, N), dtype=BITS[dtype])
    r = np.zeros(M, dtype=np.float64)
    rc = L.oracle_rmsnorm_fwd(x.ctypes.data, w.ctypes.data, y.ctypes.data,
                              r.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), None, M, N, eps,
                              offset, CODE[dtype], 0, M)
    assert rc == 0
    return y, r


def _encode(L, dtype, vals):
    vals = np.ascontiguousarray(vals, dtype=np.float64)
    out = np.zeros(vals.size, dtype=BITS[dtype])
    L.oracle_encode(CODE[dtype], vals.size, vals.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                    out.ctypes.data)
    return out


def _decode(L, dtype, bits):
    bits = np.ascontiguousarray(bits, dtype=BITS[dtype])
    out = np.zeros(bits.size, dtype=np.float64)
    L.oracle_decode(CODE[dtype], bits.size, bits.ctypes.data,
                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def _bits(dtype, values):
    return np.array([round_exact(dtype, Fraction(float(v))) for v in values], dtype=BITS[dtype])


def _patterns(dtype):
    """Finite non-negative patterns: all of them for 16-bit formats; for fp32,
    every exponent with a few fractions plus the subnormal ends."""
    if dtype != "fp32":
        return np.arange(0x7F80 if dtype == "bf16" else 0x7C00, dtype=np.uint16)
    expo = np.arange(255, dtype=np.uint32) << 23
    fr = np.array([0, 1, 3, 0x2AAAAA, 0x400000, 0x7FFFFF], dtype=np.uint32)
    sub = np.concatenate([np.arange(0, 512, dtype=np.uint32),
                          np.arange((1 << 23) - 512, 1 << 23, dtype=np.uint32)])
    return np.unique(np.concatenate([(expo[:, None] | fr[None, :]).ravel(), sub]))


def _pins_hold(L) -> bool:
    """A compact battery drawn from the oracle pins: exact rationals on random
    tiny rows (both dtypes, both offsets, several eps), constant rows at
    non-power-of-two N, and round-to-nearest-even at every bf16/fp16 midpoint
    between 1 and 2."""
    rng = np.random.default_rng(3)
    for dtype in ("bf16", "fp16", "fp32"):
        for N in (1, 3, 7, 12, 33):
            M = 3
            x = _bits(dtype, rng.normal(0, 1.5, M * N).astype(np.float32)).reshape(M, N)
            w = _bits(dtype, rng.normal(0, 0.7, N).astype(np.float32))
            for eps, offset in ((0.0, 0.0), (1e-5, 1.0), (0.25, 0.0)):
                y, r = _fwd(L, x, w, eps, offset, dtype)
                wv = [decode_exact(dtype, int(b)) for b in w]
                for i in range(M):
                    xv = [decode_exact(dtype, int(b)) for b in x[i]]
                    rr, ys = rmsnorm_row_exact(xv, wv, Fraction(float(np.float32(eps))),
                                               Fraction(offset))
                    if rr is None:
                        continue
                    if not math.isclose(r[i], float(rr), rel_tol=1e-14):
                        return False
                    for j, v in enumerate(ys):
                        got = decode_exact(dtype, int(y[i, j]))
                        if v == 0:
                            if got != 0:
                                return False
                        elif int(y[i, j]) != round_exact(dtype, v):
                            return False
        # constant rows: r = 1/sqrt(c^2 + eps) at a non-power-of-two N
        c = 0.5
        x = np.full((1, 1000), _bits(dtype, [c])[0], dtype=BITS[dtype])
        w = _bits(dtype, [1.0] * 1000)
        _, r = _fwd(L, x, w, 1e-6, 0.0, dtype)
        if not math.isclose(r[0], 1 / math.sqrt(c * c + float(np.float32(1e-6))), rel_tol=1e-14):
            return False
        # ties to even at midpoints in [1, 2) (every one for 16-bit formats)
        mbits = {"bf16": 7, "fp16": 10, "fp32": 23}[dtype]
        k = np.arange(1 << mbits, dtype=np.float64) if mbits < 16 else \
            np.unique(rng.integers(0, 1 << mbits, 4096)).astype(np.float64)
        mids = 1.0 + (k + 0.5) / (1 << mbits)
        want = [round_exact(dtype, Fraction(float(m))) for m in mids]
        if _encode(L, dtype, mids).tolist() != want:
            return False
        # finite patterns decode to their exact values and round-trip through the encoder
        pats = _patterns(dtype)
        vals = np.array([float(decode_exact(dtype, int(b))) for b in pats])
        if not np.array_equal(_decode(L, dtype, pats), vals):
            return False
        if not np.array_equal(_encode(L, dtype, vals), pats):
            return False
        # a product just below a tie rounds down (one rounding, not two)
        if not _just_below_tie_rounds_down(L, dtype):
            return False
    return True


def _just_below_tie_rounds_down(L, dtype) -> bool:
    # x = (1, 1, 1, 1), eps = 2^-30: rstd = 1/sqrt(1 + 2^-30), just under 1. With
    # offset 1 and w = 3 ulp/2 the exact y sits 2^-31 below the midpoint between
    # 1 + 1 ulp (odd) and 1 + 2 ulp (even): it must round down to 1 + 1 ulp,
    # while rounding through fp32 first lands on the midpoint and goes up.
    ulp = {"bf16": 2.0 ** -7, "fp16": 2.0 ** -10, "fp32": 2.0 ** -23}[dtype]
    x = _bits(dtype, [1.0] * 4).reshape(1, 4)
    w = _bits(dtype, [1.5 * ulp] * 4)
    y, _ = _fwd(L, x, w, 2.0 ** -30, 1.0, dtype)
    return y[0].tolist() == [round_exact(dtype, Fraction(1) + Fraction(ulp))] * 4


# Slips in the backward (dx = r (dy s - x r^2 c / N), c = sum dy s x, dw = sum dy x r).
BWD_MUTATIONS = {
    "bwd: projection term dropped": ("double v = r * (gv * sv - xv * r * r * c / (double)N);",
                                     "double v = r * gv * sv;"),
    "bwd: projection term added": ("double v = r * (gv * sv - xv * r * r * c / (double)N);",
                                   "double v = r * (gv * sv + xv * r * r * c / (double)N);"),
    "bwd: r instead of r^2": ("double v = r * (gv * sv - xv * r * r * c / (double)N);",
                              "double v = r * (gv * sv - xv * r * c / (double)N);"),
    "bwd: divides by N+1": ("double v = r * (gv * sv - xv * r * r * c / (double)N);",
                            "double v = r * (gv * sv - xv * r * r * c / (double)(N + 1));"),
    "bwd: weight left out of c": (
        "c += load_elem(dtype, dy, base + j) * (off + load_elem(dtype, w, j)) *",
        "c += load_elem(dtype, dy, base + j) * (off + 1.0) *"),
    "bwd: offset left out of the scale": ("double sv = off + load_elem(dtype, w, j);",
                                          "double sv = load_elem(dtype, w, j);"),
    "bwd: dw without r": ("if (dw) dw[j] += gv * xv * r;", "if (dw) dw[j] += gv * xv;"),
    "bwd: dw times the scale": ("if (dw) dw[j] += gv * xv * r;",
                                "if (dw) dw[j] += gv * xv * r * sv;"),
    "bwd: recomputed rstd without eps": ("r = 1.0 / sqrt(s / (double)N + (double)eps);",
                                         "r = 1.0 / sqrt(s / (double)N);"),
    "bwd: x and dy swapped": (
        "double xv = load_elem(dtype, x, base + j), gv = load_elem(dtype, dy, base + j);",
        "double gv = load_elem(dtype, x, base + j), xv = load_elem(dtype, dy, base + j);"),
}


def _bwd(L, x, w, dy, rstd, eps, offset, dtype):
    M, N = x.shape
    x, w, dy = (np.ascontiguousarray(a, dtype=BITS[dtype]) for a in (x, w, dy))
    dx = np.zeros((M, N), dtype=BITS[dtype])
    dx64 = np.zeros((M, N), dtype=np.float64)
    dw = np.zeros(N, dtype=np.float64)
    f64p = ctypes.POINTER(ctypes.c_double)
    rp = None if rstd is None else np.ascontiguousarray(rstd, dtype=np.float64)
    rc = L.oracle_rmsnorm_bwd(x.ctypes.data, w.ctypes.data, dy.ctypes.data,
                              None if rp is None else rp.ctypes.data_as(f64p), dx.ctypes.data,
                              dx64.ctypes.data_as(f64p), dw.ctypes.data_as(f64p), M, N, eps,
                              offset, CODE[dtype])
    assert rc == 0
    return dx, dx64, dw


def _bwd_pins_hold(L) -> bool:
    """The backward against torch float64 autograd of the textbook forward
    expression (an outside routine), with the saved rstd passed in and with
    rstd recomputed; dx's stored bits are the encoder's rounding of its fp64
    value."""
    import torch
    rng = np.random.default_rng(5)
    eps = 1e-3
    e = float(np.float32(eps))
    for dtype in ("bf16", "fp16", "fp32"):
        for N in (1, 5, 33):
            M = 3
            x = _bits(dtype, rng.normal(0, 1.5, M * N).astype(np.float32)).reshape(M, N)
            dy = _bits(dtype, rng.normal(0, 1.0, M * N).astype(np.float32)).reshape(M, N)
            w = _bits(dtype, rng.normal(0, 0.7, N).astype(np.float32))
            xv = torch.tensor(_decode(L, dtype, x).reshape(M, N), requires_grad=True)
            gv = torch.tensor(_decode(L, dtype, dy).reshape(M, N))
            for offset in (0.0, 1.0):
                wv = torch.tensor(_decode(L, dtype, w), requires_grad=True)
                xv.grad = None
                r = torch.rsqrt(xv.pow(2).mean(-1, keepdim=True) + e)
                ((xv * r * (offset + wv)) * gv).sum().backward()
                terms = (r * gv.abs() * (offset + wv).abs()).detach().numpy()
                r64 = r.detach().numpy().ravel()
                for rstd in (r64, None):
                    dx, dx64, dw = _bwd(L, x, w, dy, rstd, eps, offset, dtype)
                    if not np.all(np.abs(dx64 - xv.grad.numpy())
                                  <= 1e-11 * np.abs(dx64) + 1e-13 * terms):
                        return False
                    ref_dw = wv.grad.numpy()
                    if not np.allclose(dw, ref_dw, rtol=1e-11, atol=1e-13 * np.abs(ref_dw).max()):
                        return False
                    if not np.array_equal(dx.ravel(), _encode(L, dtype, dx64.ravel())):
                        return False
    return True


def test_the_oracle_itself_passes_the_battery(tmp_path):
    assert _pins_hold(_build(str(tmp_path), open(SRC).read()))


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_each_planted_slip_fails_the_pins(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor not found: {old}"
    # The first occurrence is the forward's (the backward follows it in the file).
    assert not _pins_hold(_build(str(tmp_path), src.replace(old, new, 1)))


def test_the_oracle_backward_passes_its_battery(tmp_path):
    assert _bwd_pins_hold(_build(str(tmp_path), open(SRC).read()))


@pytest.mark.parametrize("name", list(BWD_MUTATIONS))
def test_each_planted_backward_slip_fails_the_pins(tmp_path, name):
    old, new = BWD_MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old}"
    assert not _bwd_pins_hold(_build(str(tmp_path), src.replace(old, new)))
