"""GPU parity of the backward (dx, dw) against the oracle's fp64 backward, on the
same seeded inputs and the same fp32 rstd (the oracle forward's, rounded to
fp32: the value a forward keeps for the backward).

bf16, fp16 and fp32 inputs. Tolerance, derived from the arithmetic: dx = r (dy s - x r^2 c / N) is a
difference of two fp32 terms, each with relative error of a few 1e-7 (c is a
fp32 sum over the row), so |dx_gpu - dx| <= 1 ulp(dx) + 1e-5 * r (|dy s| +
|x| r^2 sum|dy s x| / N); dw is an fp32 sum over rows (per CTA, then over
CTAs), so |dw_gpu - dw| <= 1e-5 * sum_i |dy x r|.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TAU = 1e-5
DT = {"bf16": B.BF16, "fp16": B.FP16, "fp32": B.FP32}


def _ulp(dtype, v):
    mbits, emin = {"bf16": (7, -126), "fp16": (10, -14), "fp32": (23, -126)}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-300)))
    return np.exp2(np.maximum(e, emin) - mbits)


def _inputs(M, N, dtype, seed, offset=0.0):
    wl = W.custom(M, N, dtype, seed=seed, offset=offset)
    x, w = W.generate(wl)
    g = W.custom(M, N, dtype, seed=seed + 1000)
    dy, _ = W.generate(g)
    _, r64 = oracle.rmsnorm_fwd(x, w, wl.eps, offset, dtype)
    rstd = r64.astype(np.float32)
    return x, w, dy, rstd


def _check(x, w, dy, rstd, dx_bits, dw, offset, dtype, where=""):
    _, dx64, dw64 = oracle.rmsnorm_bwd(x, w, dy, offset, dtype, rstd=rstd.astype(np.float64))
    xv, gv = oracle.decode(dtype, x), oracle.decode(dtype, dy)
    sv = offset + oracle.decode(dtype, w)
    r = rstd.astype(np.float64)[:, None]
    cabs = np.abs(gv * sv * xv).sum(axis=1, keepdims=True)
    bound = _ulp(dtype, dx64) + TAU * r * (np.abs(gv * sv) + np.abs(xv) * r * r * cabs / x.shape[1])
    err = np.abs(oracle.decode(dtype, dx_bits) - dx64)
    assert np.all(err <= bound), f"{where}: dx off by {np.max(err / bound):.3g} of the bound"
    dwb = TAU * (np.abs(gv * xv) * r).sum(axis=0) + 1e-30
    errw = np.abs(dw.astype(np.float64) - dw64)
    assert np.all(errw <= dwb), f"{where}: dw off by {np.max(errw / dwb):.3g} of the bound"


def _run(x, w, dy, rstd, offset, dtype, inplace=None, **opts):
    M, N = x.shape
    xd = W.to_torch(x, dtype).cuda()
    wd = W.to_torch(w, dtype).cuda()
    gd = W.to_torch(dy, dtype).cuda()
    rd = torch.from_numpy(rstd).cuda()
    dxd = xd if inplace == "x" else gd if inplace == "dy" else torch.empty_like(xd)
    dwd = torch.full((N,), -7.0, dtype=torch.float32, device="cuda")
    o = B.make_options(**opts) if opts else None
    nbytes = B.rmsnorm_bwd_workspace_size(M, N, DT[dtype], o)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    rc = B.rmsnorm_bwd(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), gd.data_ptr(), dxd.data_ptr(),
                       dwd.data_ptr(), M, N, offset, DT[dtype], ws.data_ptr(), ws.numel() * 4, o,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    torch.cuda.synchronize()
    return W.from_torch(dxd), dwd.cpu().numpy()


SHAPES = [(1, 8), (37, 512), (300, 1000), (64, 4096), (33, 8192), (17, 16384), (9, 777),
          (5, 20000), (130, 520)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("variant", ["auto", "warp", "cta", "tma", "generic"])
def test_bwd_parity(dtype, M, N, variant):
    offset = float((M + N) % 2)
    x, w, dy, rstd = _inputs(M, N, dtype, seed=M * 7 + N, offset=offset)
    try:
        B.rmsnorm_bwd_workspace_size(M, N, DT[dtype], B.make_options(variant=variant))
    except B.RMSNormError as e:
        assert e.status == -8
        pytest.skip("variant does not take this shape")
    for max_ctas in (0, 3):
        try:
            dx, dw = _run(x, w, dy, rstd, offset, dtype, variant=variant, max_ctas=max_ctas)
        except AssertionError:
            e = 4 if dtype == "fp32" else 8   # elements per 16-byte vector
            nvec = N // e                      # vector kernels: up to 2048 (CTA), 128 (warp)
            if (variant == "cta" and (N % e or nvec > 2048)) or \
                    (variant == "warp" and (N % e or nvec > 128)) or \
                    (variant == "tma" and (N % e or nvec > 1024)):
                pytest.skip("vector kernel does not take this shape")
            raise
        _check(x, w, dy, rstd, dx, dw, offset, dtype, where=f"{variant} {M}x{N} {max_ctas}")


@pytest.mark.parametrize("M,N,dtype", [(64, 100000, "bf16"), (7, 70001, "fp32"), (300, 60000, "fp16")])
@pytest.mark.parametrize("max_ctas", [0, 5])
def test_bwd_rows_past_the_shared_memory_limit(M, N, dtype, max_ctas):
    # Rows whose fp32 dw partial does not fit in shared memory (N * 4 bytes
    # past ~227 KB): the general kernel keeps the partial in its workspace row.
    offset = float(N % 2)
    x, w, dy, rstd = _inputs(M, N, dtype, seed=N + M, offset=offset)
    plan_bytes = B.rmsnorm_bwd_workspace_size(M, N, DT[dtype], B.make_options(max_ctas=max_ctas))
    assert plan_bytes % (N * 4) == 0 and plan_bytes <= 64 << 20
    dx, dw = _run(x, w, dy, rstd, offset, dtype, max_ctas=max_ctas)
    _check(x, w, dy, rstd, dx, dw, offset, dtype, where=f"{M}x{N} {dtype} {max_ctas}")


@pytest.mark.parametrize("inplace", ["x", "dy"])
@pytest.mark.parametrize("N", [512, 777])
def test_bwd_in_place(inplace, N):
    x, w, dy, rstd = _inputs(200, N, "bf16", seed=N + 1, offset=1.0)
    dx, dw = _run(x, w, dy, rstd, 1.0, "bf16", inplace=inplace)
    _check(x, w, dy, rstd, dx, dw, 1.0, "bf16")


@pytest.mark.parametrize("name", ["rmsnorm_16384x512_bf16", "rmsnorm_32768x1000_bf16_gemma"])
def test_bwd_full_size_workloads(name):
    wl = W.WORKLOADS[name]
    x, w = W.generate(wl)
    dy, _ = W.generate(W.custom(wl.M, wl.N, wl.dtype, seed=99))
    _, r64 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, wl.dtype)
    rstd = r64.astype(np.float32)
    dx, dw = _run(x, w, dy, rstd, wl.offset, wl.dtype)
    _check(x, w, dy, rstd, dx, dw, wl.offset, wl.dtype, where=name)


def test_bwd_is_deterministic_and_m_zero_zeroes_dw():
    x, w, dy, rstd = _inputs(3000, 1024, "fp16", seed=5)
    a = _run(x, w, dy, rstd, 0.0, "fp16")
    b = _run(x, w, dy, rstd, 0.0, "fp16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    wd = W.to_torch(w, "fp16").cuda()
    dwd = torch.full((1024,), 3.0, dtype=torch.float32, device="cuda")
    assert B.rmsnorm_bwd(0, wd.data_ptr(), 0, 0, 0, dwd.data_ptr(), 0, 1024, 0.0, B.FP16, 0, 0, None,
                         torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(dwd) == 0


def test_bwd_rejects_a_small_workspace():
    M, N = 64, 512
    xd = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    rd = torch.ones(M, dtype=torch.float32, device="cuda")
    dwd = torch.zeros(N, dtype=torch.float32, device="cuda")
    need = B.rmsnorm_bwd_workspace_size(M, N, B.BF16)
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    rc = B.rmsnorm_bwd(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), xd.data_ptr(), xd.data_ptr(),
                       dwd.data_ptr(), M, N, 0.0, B.BF16, ws.data_ptr(), 16, None,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == -11


def test_fp32_full_size_and_in_place():
    x, w, dy, rstd = _inputs(32768, 1000, "fp32", seed=21, offset=1.0)
    dx, dw = _run(x, w, dy, rstd, 1.0, "fp32")
    _check(x, w, dy, rstd, dx, dw, 1.0, "fp32", where="fp32 32768x1000")
    dx2, dw2 = _run(x, w, dy, rstd, 1.0, "fp32", inplace="dy")
    assert np.array_equal(dx, dx2) and np.array_equal(dw, dw2)


def test_torch_convenience_forward_then_backward():
    x, w, dy, _ = _inputs(500, 2048, "bf16", seed=8, offset=1.0)
    xd, wd, gd = (W.to_torch(a, "bf16").cuda() for a in (x, w, dy))
    y, rstd = B.fwd(xd, wd, eps=1e-6, offset=1.0)
    dx, dw = B.bwd(xd, wd, rstd, gd, offset=1.0)
    torch.cuda.synchronize()
    # The GPU forward's rstd is within 1e-5 of the oracle's: check the backward
    # against the oracle fed the oracle's own rstd, with the tolerance widened by
    # that difference (dx and dw are first order in r).
    _, r64 = oracle.rmsnorm_fwd(x, w, 1e-6, 1.0, "bf16")
    _, dx64, dw64 = oracle.rmsnorm_bwd(x, w, dy, 1.0, "bf16", rstd=r64)
    got = oracle.decode("bf16", W.from_torch(dx))
    assert np.all(np.abs(got - dx64) <= _ulp("bf16", dx64) + 3e-5 * np.abs(dx64).max())
    assert np.allclose(dw.cpu().numpy(), dw64, rtol=1e-4, atol=1e-4 * np.abs(dw64).max())


def _bwd_call(xd, wd, rd, gd, dxd, dwd, offset, dtype, ws, **opts):
    M, N = xd.shape
    rc = B.rmsnorm_bwd(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), gd.data_ptr(), dxd.data_ptr(),
                       dwd.data_ptr(), M, N, offset, DT[dtype], ws.data_ptr(), ws.numel() * 4,
                       B.make_options(**opts), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()


@pytest.mark.parametrize("variant,M,N,dtype", [("warp", 3000, 512, "bf16"), ("warp", 777, 1000, "fp16"),
                                               ("cta", 2000, 4096, "bf16"), ("cta", 300, 2048, "fp32"),
                                               ("tma", 3000, 512, "bf16"), ("tma", 500, 4096, "fp16"),
                                               ("tma", 777, 1000, "fp32"), ("auto", 5000, 768, "bf16")])
def test_bwd_early_loads_chain(variant, M, N, dtype):
    # With RMSNORM_FLAG_EARLY_LOADS the caller promises only that x, w and rstd
    # are not written by the kernel before; dy may be. A chain where each call's
    # dy is the previous call's dx, launched back to back, must give the bits
    # of the same calls with the device synchronised between them; and each
    # first call (whose inputs come from the generator) matches the oracle.
    x, w, dy, rstd = _inputs(M, N, dtype, seed=N + M + 5, offset=1.0)
    xd, wd, rd = W.to_torch(x, dtype).cuda(), W.to_torch(w, dtype).cuda(), torch.from_numpy(rstd).cuda()
    nbytes = B.rmsnorm_bwd_workspace_size(M, N, DT[dtype], B.make_options(variant=variant))
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    steps = 4
    outs = {}
    for early in (False, True):
        g = [W.to_torch(dy, dtype).cuda()] + [torch.empty_like(xd) for _ in range(steps)]
        dws = [torch.empty(N, dtype=torch.float32, device="cuda") for _ in range(steps)]
        for k in range(steps):
            _bwd_call(xd, wd, rd, g[k], g[k + 1], dws[k], 1.0, dtype, ws, variant=variant,
                      early_loads=early)
            if not early:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        outs[early] = ([W.from_torch(t) for t in g[1:]], [d.cpu().numpy() for d in dws])
    for k in range(steps):
        assert np.array_equal(outs[True][0][k], outs[False][0][k]), f"dx differs at step {k}"
        assert np.array_equal(outs[True][1][k], outs[False][1][k]), f"dw differs at step {k}"
    _check(x, w, dy, rstd, outs[True][0][0], outs[True][1][0], 1.0, dtype, where="first call")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("N", [8, 512, 1000, 4096, 8192])
@pytest.mark.parametrize("rows,stages", [(1, 1), (3, 2), (8, 3), (16, 2), (0, 0)])
def test_bwd_tma_stage_shapes(dtype, N, rows, stages):
    # The staged backward over stage shapes, grids small enough that every CTA
    # walks many chunks (ragged last chunk: M is not a multiple of the rows per
    # stage), and in place (dx == x, dx == dy).
    e = 4 if dtype == "fp32" else 8
    if N // e > 1024:
        pytest.skip("the staged kernel takes rows of up to 16 KB")
    M = 203
    opts = dict(variant="tma", rows_per_stage=rows, stages=stages)
    try:
        B.rmsnorm_bwd_plan_info(M, N, DT[dtype], B.make_options(**opts))
    except B.RMSNormError as err:
        assert err.status == -8
        pytest.skip("the stages do not fit in shared memory")
    x, w, dy, rstd = _inputs(M, N, dtype, seed=N + rows + stages, offset=float(rows % 2))
    for max_ctas in (0, 1, 5):
        dx, dw = _run(x, w, dy, rstd, float(rows % 2), dtype, max_ctas=max_ctas, **opts)
        _check(x, w, dy, rstd, dx, dw, float(rows % 2), dtype, where=f"{N} {rows}x{stages} {max_ctas}")
    for inplace in ("x", "dy"):
        dx, dw = _run(x, w, dy, rstd, float(rows % 2), dtype, inplace=inplace, max_ctas=3, **opts)
        _check(x, w, dy, rstd, dx, dw, float(rows % 2), dtype, where=f"{N} in place {inplace}")


def test_bwd_tma_bounded_wait_reports_timeout_and_recovers():
    # A 1 ns wait bound makes the first stage's wait give up before its copies
    # land: the kernel records the timeout, waits for its own copies and exits;
    # the status call reports it once, and the next normal call is exact.
    M, N, dtype = 4096, 1024, "bf16"
    x, w, dy, rstd = _inputs(M, N, dtype, seed=21)
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_check_device_status(s) == 0
    _run(x, w, dy, rstd, 0.0, dtype, variant="tma", wait_limit_ns=1)
    assert B.rmsnorm_check_device_status(s) == -7
    assert B.rmsnorm_check_device_status(s) == 0
    dx, dw = _run(x, w, dy, rstd, 0.0, dtype, variant="tma")
    assert B.rmsnorm_check_device_status(s) == 0
    _check(x, w, dy, rstd, dx, dw, 0.0, dtype, where="after timeout")


@pytest.mark.parametrize("variant", ["warp", "cta"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("M,N", [(37, 512), (300, 1000), (64, 4096), (130, 520)])
@pytest.mark.parametrize("PW", [1, 4, 15])
def test_bwd_prewait_prefetch_parity(variant, dtype, M, N, PW):
    # Rows of x and dy asked into L2 before the wait for the previous kernel: a
    # hint only, so dx and dw must still match the oracle, for strict order and
    # early loads, the full grid and a grid of three CTAs walking every row.
    e = 4 if dtype == "fp32" else 8
    if variant == "warp" and N // e > 128:
        pytest.skip("the warp kernel takes rows of up to 128 vectors")
    x, w, dy, rstd = _inputs(M, N, dtype, seed=M + N + PW, offset=1.0)
    plan = B.rmsnorm_bwd_plan_info(M, N, DT[dtype], B.make_options(variant=variant, prewait_prefetch=PW))
    assert plan["prewait_prefetch"] == PW
    for max_ctas in (0, 3):
        for early in (False, True):
            dx, dw = _run(x, w, dy, rstd, 1.0, dtype, variant=variant, max_ctas=max_ctas,
                          prewait_prefetch=PW, early_loads=early)
            _check(x, w, dy, rstd, dx, dw, 1.0, dtype, where=f"{variant} {M}x{N} PW {PW}")


def test_bwd_automatic_prewait_plan():
    # The row kernels prefetch one row of x and dy per warp (CTA) before the
    # wait by default; none without PDL or when the caller says -1; the staged
    # and general kernels take none.
    for N, dtype in ((512, "bf16"), (4096, "bf16"), (512, "fp32")):
        assert B.rmsnorm_bwd_plan_info(16384, N, DT[dtype])["prewait_prefetch"] == 1
        assert B.rmsnorm_bwd_plan_info(16384, N, DT[dtype], B.make_options(pdl=False))["prewait_prefetch"] == 0
        assert B.rmsnorm_bwd_plan_info(16384, N, DT[dtype],
                                       B.make_options(prewait_prefetch=-1))["prewait_prefetch"] == 0
    assert B.rmsnorm_bwd_plan_info(16384, 512, DT["bf16"],
                                   B.make_options(variant="tma"))["prewait_prefetch"] == 0
    assert B.rmsnorm_bwd_plan_info(100, 70001, DT["fp32"])["prewait_prefetch"] == 0


@pytest.mark.parametrize("variant,M,N,dtype", [("warp", 16384, 512, "bf16"), ("cta", 4000, 4096, "bf16"),
                                               ("warp", 8000, 512, "fp32")])
@pytest.mark.parametrize("PW", [0, 2])
def test_bwd_prewait_chain_keeps_stream_order(variant, M, N, dtype, PW):
    # Each call's dy is the previous call's dx, launched back to back under
    # strict order with the pre-wait prefetch (and the reduction letting the
    # next row kernel start early): the bits of the same calls with the device
    # synchronised between them.
    x, w, dy, rstd = _inputs(M, N, dtype, seed=N + M + PW, offset=0.0)
    xd, wd, rd = W.to_torch(x, dtype).cuda(), W.to_torch(w, dtype).cuda(), torch.from_numpy(rstd).cuda()
    o = B.make_options(variant=variant, prewait_prefetch=PW)
    assert B.rmsnorm_bwd_plan_info(M, N, DT[dtype], o)["prewait_prefetch"] == (PW or 1)
    nbytes = B.rmsnorm_bwd_workspace_size(M, N, DT[dtype], o)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    steps = 4
    outs = {}
    for sync in (False, True):
        g = [W.to_torch(dy, dtype).cuda()] + [torch.empty_like(xd) for _ in range(steps)]
        dws = [torch.empty(N, dtype=torch.float32, device="cuda") for _ in range(steps)]
        for k in range(steps):
            _bwd_call(xd, wd, rd, g[k], g[k + 1], dws[k], 0.0, dtype, ws, variant=variant,
                      prewait_prefetch=PW)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        outs[sync] = ([W.from_torch(t) for t in g[1:]], [d.cpu().numpy() for d in dws])
    for k in range(steps):
        assert np.array_equal(outs[True][0][k], outs[False][0][k]), f"dx differs at step {k}"
        assert np.array_equal(outs[True][1][k], outs[False][1][k]), f"dw differs at step {k}"
    _check(x, w, dy, rstd, outs[False][0][0], outs[False][1][0], 0.0, dtype, where="first call")
