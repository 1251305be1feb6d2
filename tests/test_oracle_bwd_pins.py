"""Pins for the oracle's backward (derived by the chain rule; the pages only say
rstd is kept "for backward").

The backward is pinned to things outside the oracle: torch float64 autograd of
the textbook forward expression, central finite differences in plain Python,
closed forms and invariants that follow from the forward's scale invariance.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import workloads as W


def _rand(rng, shape, dtype, scale=1.0):
    t = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
    return W.from_torch(t.to(torch.bfloat16 if dtype == "bf16" else torch.float16))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("offset", [0.0, 1.0])
@pytest.mark.parametrize("N", [1, 7, 64, 1000])
def test_backward_matches_torch_float64_autograd(dtype, offset, N):
    rng = np.random.default_rng(N + int(offset))
    M = 9
    x, dy = _rand(rng, (M, N), dtype, 2.0), _rand(rng, (M, N), dtype)
    w = _rand(rng, (N,), dtype, 0.4)
    eps = 1e-5
    e = float(np.float32(eps))
    xt = W.to_torch(x, dtype).to(torch.float64).requires_grad_(True)
    wt = W.to_torch(w, dtype).to(torch.float64).requires_grad_(True)
    gt = W.to_torch(dy, dtype).to(torch.float64)
    y = xt * torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + e) * (offset + wt)
    (y * gt).sum().backward()
    _, dx64, dw = oracle.rmsnorm_bwd(x, w, dy, offset, dtype, eps=eps)
    # dx is a difference of two terms of size r |dy s|; it can cancel (at N = 1
    # almost entirely), so the absolute tolerance scales with the terms.
    with torch.no_grad():
        r = torch.rsqrt(xt.pow(2).mean(-1, keepdim=True) + e)
        terms = (r * gt.abs() * (offset + wt).abs()).numpy()
    assert np.all(np.abs(dx64 - xt.grad.numpy()) <= 1e-11 * np.abs(dx64) + 1e-13 * terms)
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-13 * np.abs(dw).max())


def test_backward_matches_central_differences():
    # Pure Python fp64: L(x, w) = sum dy * y, derivative by central differences.
    rng = np.random.default_rng(2)
    M, N, eps, offset = 2, 5, 1e-3, 1.0
    x = _rand(rng, (M, N), "bf16")
    w = _rand(rng, (N,), "bf16", 0.5)
    dy = _rand(rng, (M, N), "bf16")
    X, Wv, G = (oracle.decode("bf16", a).tolist() for a in (x, w, dy))
    e = float(np.float32(eps))

    def loss(Xv, Wl):
        tot = 0.0
        for i in range(M):
            r = 1.0 / math.sqrt(sum(v * v for v in Xv[i]) / N + e)
            tot += sum(G[i][j] * Xv[i][j] * r * (offset + Wl[j]) for j in range(N))
        return tot

    _, dx64, dw = oracle.rmsnorm_bwd(x, w, dy, offset, "bf16", eps=eps)
    h = 1e-6
    for i in range(M):
        for j in range(N):
            Xp = [row[:] for row in X]
            Xm = [row[:] for row in X]
            Xp[i][j] += h
            Xm[i][j] -= h
            fd = (loss(Xp, Wv) - loss(Xm, Wv)) / (2 * h)
            assert dx64[i, j] == pytest.approx(fd, rel=1e-6, abs=1e-8)
    for j in range(N):
        Wp, Wm = Wv[:], Wv[:]
        Wp[j] += h
        Wm[j] -= h
        fd = (loss(X, Wp) - loss(X, Wm)) / (2 * h)
        assert dw[j] == pytest.approx(fd, rel=1e-6, abs=1e-8)


def test_constant_rows_have_zero_dx_at_eps_zero():
    # y = sign(c) (offset + w) does not depend on |c| when eps = 0, so with a
    # constant upstream gradient dx vanishes exactly and dw_j = sum_i d_i sign(c_i).
    N = 12
    cs, ds = [1.5, -0.25, 3.0], [0.5, -2.0, 1.0]
    x = np.array([[oracle.encode("bf16", np.array([c]))[0]] * N for c in cs], dtype=np.uint16)
    dy = np.array([[oracle.encode("bf16", np.array([d]))[0]] * N for d in ds], dtype=np.uint16)
    w = oracle.encode("bf16", np.ones(N))
    _, dx64, dw = oracle.rmsnorm_bwd(x, w, dy, 0.0, "bf16", eps=0.0)
    assert np.all(np.abs(dx64) <= 1e-15)
    want = sum(d * math.copysign(1.0, c) for c, d in zip(cs, ds))
    assert np.allclose(dw, want, rtol=1e-15)


@pytest.mark.parametrize("k", [-3, 2])
def test_scale_invariance_of_the_gradients(k):
    # eps = 0: y(alpha x) = y(x), so dx(alpha x) = dx(x) / alpha and dw unchanged, exactly
    # for alpha a power of two.
    rng = np.random.default_rng(30 + k)
    mag = rng.uniform(0.5, 2.0, (4, 33)) * rng.choice([-1.0, 1.0], (4, 33))
    x = W.from_torch(torch.from_numpy(mag).to(torch.bfloat16))
    xs = W.from_torch(torch.from_numpy(mag).to(torch.bfloat16).to(torch.float64).mul(2.0 ** k)
                      .to(torch.bfloat16))
    dy, w = _rand(rng, (4, 33), "bf16"), _rand(rng, (33,), "bf16")
    _, a, da = oracle.rmsnorm_bwd(x, w, dy, 1.0, "bf16", eps=0.0)
    _, b, db = oracle.rmsnorm_bwd(xs, w, dy, 1.0, "bf16", eps=0.0)
    assert np.array_equal(b, a / 2.0 ** k) and np.array_equal(db, da)


def test_gradient_is_orthogonal_to_x_at_eps_zero():
    # Scale invariance again: sum_j dx_ij x_ij = r c (1 - r^2 ms) = 0 when eps = 0.
    rng = np.random.default_rng(4)
    x, dy, w = _rand(rng, (6, 257), "bf16"), _rand(rng, (6, 257), "bf16"), _rand(rng, (257,), "bf16")
    _, dx64, _ = oracle.rmsnorm_bwd(x, w, dy, 0.0, "bf16", eps=0.0)
    xv = oracle.decode("bf16", x)
    dots = (dx64 * xv).sum(axis=1)
    assert np.all(np.abs(dots) <= 1e-12 * np.abs(dx64).sum(axis=1) * np.abs(xv).max())


def test_saved_rstd_equals_recomputed():
    rng = np.random.default_rng(5)
    x, dy, w = _rand(rng, (5, 100), "fp16", 30.0), _rand(rng, (5, 100), "fp16"), _rand(rng, (100,), "fp16")
    _, r = oracle.rmsnorm_fwd(x, w, 1e-6, 0.0, "fp16")
    a = oracle.rmsnorm_bwd(x, w, dy, 0.0, "fp16", rstd=r)
    b = oracle.rmsnorm_bwd(x, w, dy, 0.0, "fp16", eps=1e-6)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
    # and dx is the single rounding of its fp64 value
    assert np.array_equal(a[0], oracle.encode("fp16", a[1]))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_constant_row_centres_the_scaled_gradient(dtype, offset):
    # Closed form: x_ij = c for all j, eps = 0 gives r = 1/|c| and
    # x_j r^2 c_i / N = mean_k(dy_k s_k), so dx_j = (dy_j s_j - mean_k dy_k s_k) / |c|
    # and dw_j = sum_i dy_ij sign(c_i). Dyadic inputs and N = 16 make it exact.
    rng = np.random.default_rng(17)
    N = 16
    cs = [2.0, -0.5, 4.0]
    dyv = rng.integers(-8, 9, (3, N)) / 4.0
    wv = rng.integers(-4, 5, N) / 8.0
    x = np.array([oracle.encode(dtype, np.full(N, c)) for c in cs])
    dy = oracle.encode(dtype, dyv.ravel()).reshape(3, N)
    w = oracle.encode(dtype, wv)
    _, dx64, dw = oracle.rmsnorm_bwd(x, w, dy, offset, dtype, eps=0.0)
    g = dyv * (offset + wv)
    want = (g - g.mean(axis=1, keepdims=True)) / np.abs(np.array(cs))[:, None]
    assert np.array_equal(dx64, want)
    assert np.array_equal(dw, (dyv * np.sign(np.array(cs))[:, None]).sum(axis=0))
