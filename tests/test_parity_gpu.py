"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs (y within 1 ulp, rstd within 1e-5 relative).

Covers the five named workloads at full size in the automatic launch
configuration (the one the benchmark times), every kernel variant on shapes
that span several tiles with ragged tails, forced small grids (many rows per
CTA), every lanes-per-row / stage setting the variants take, odd N and
misaligned pointers, in-place calls, M = 0, zero rows, canaries around every
buffer, element counts past 2^31, and the bounded-wait timeout path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W
from parity_util import (DT, DeviceCase, compare, compare_blocked, compare_fp32, oracle_rows,
                         oracle_threaded, sample_rows)

pytestmark = pytest.mark.gpu


def _plan(M, N, dtype, case=None, **opts):
    x = case.x.data_ptr() if case else 0
    w = case.w.data_ptr() if case else 0
    y = case.y.data_ptr() if case else 0
    return B.rmsnorm_plan_info(M, N, DT[dtype], x, w, y, B.make_options(**opts) if opts else None)


def _run_and_check(x, w, dtype, eps, offset, rows=None, x_shift=0, y_shift=0, inplace=False,
                   expect_variant=None, **opts):
    case = DeviceCase(x, w, dtype, x_shift=x_shift, y_shift=y_shift, inplace=inplace)
    if expect_variant is not None:
        assert _plan(x.shape[0], x.shape[1], dtype, case, **opts)["variant"] == expect_variant
    rc = case.run(eps, offset, **opts)
    assert rc == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    yo, ro = oracle_rows(x, w, eps, offset, dtype, rows)
    if rows is not None:
        y, r = y[rows], r[rows]
    return compare(y, r, yo, ro, dtype, where=f"{dtype} {x.shape} {opts}")


# ---------------------------------------------------------------- full-size workloads

_ORACLE_CACHE: dict = {}


def _full_oracle(name):
    """Inputs and the oracle's y and rstd on every row of a named workload
    (computed once per test session, threaded over the host cores)."""
    if name not in _ORACLE_CACHE:
        wl = W.WORKLOADS[name]
        x, w = W.generate(wl)
        _ORACLE_CACHE[name] = (x, w) + oracle_threaded(x, w, wl.eps, wl.offset, wl.dtype)
    return _ORACLE_CACHE[name]


@pytest.mark.parametrize("name", list(W.WORKLOADS))
@pytest.mark.parametrize("early", [False, True], ids=["strict", "early_loads"])
def test_workload_full_size_automatic_launch(name, early, parity_report):
    # The automatic plan, in both launch modes bench.py times (early loads: two
    # back-to-back calls, the second overlapping the first), compared with the
    # oracle on every element of every row.
    wl = W.WORKLOADS[name]
    x, w, yo, ro = _full_oracle(name)
    case = DeviceCase(x, w, wl.dtype)
    for _ in range(2 if early else 1):
        assert case.run(wl.eps, wl.offset, early_loads=early) == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    # Properties over every row: rstd finite and positive, y finite.
    assert np.all(np.isfinite(r)) and np.all(r > 0)
    exp_mask = 0x7F80 if wl.dtype == "bf16" else 0x7C00
    assert not np.any((y & exp_mask) == exp_mask), "non-finite y"
    max_ulp, max_rel, hist = compare_blocked(y, r, yo, ro, wl.dtype, where=name)
    plan = _plan(wl.M, wl.N, wl.dtype, case, early_loads=early)
    parity_report.append(
        f"{name} [{'early loads' if early else 'strict'}, {plan['variant']}]: {wl.M} rows x "
        f"{wl.N} compared, max ulp {max_ulp} (" +
        ", ".join(f"{k}: {v}" for k, v in sorted(hist.items())) + f"), max rstd rel err {max_rel:.3g}")
    if wl.dtype == "fp16":
        assert abs(float(np.mean(r)) * wl.x_std - 1.0) < 0.01  # rstd ~ 1/64


@pytest.mark.parametrize("M,N,dtype,max_per_sm", [(65536, 512, "bf16", 6), (131072, 512, "bf16", 3),
                                                (65536, 256, "fp32", 6), (32768, 512, "bf16", 6)])
def test_strict_warp_grid_for_many_passes(M, N, dtype, max_per_sm):
    # Under strict order the warp kernel's whole-warp teams that walk 16 passes
    # of rows or more run half the resident CTAs, and every plan here
    # prefetches its first rows into L2 before the wait; the rows are the same
    # work whatever the grid, so every row must still match.
    wl = W.custom(M, N, dtype, seed=M + N)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, dtype)
    plan = _plan(M, N, dtype, case, variant="warp")
    assert plan["variant"] == "warp" and plan["lanes_per_row"] == 32
    assert plan["grid"] <= max_per_sm * plan["sm_count"]
    assert plan["prewait_prefetch"] >= 1 and plan["l2_prefetch"] == 1
    assert case.run(wl.eps, wl.offset, variant="warp") == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    if dtype == "fp32":
        _, ro, y64 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, dtype, want_y64=True)
        compare_fp32(y, r, y64, ro, where=f"{M}x{N}")
    else:
        yo, ro = oracle_threaded(x, w, wl.eps, wl.offset, dtype)
        compare_blocked(y, r, yo, ro, dtype, where=f"{M}x{N}")


# ---------------------------------------------------------------- every variant

SHAPES = [(1, 8), (3, 64), (37, 512), (257, 1000), (64, 1024), (17, 2048), (9, 4096),
          (5, 8192), (130, 520), (11, 16384)]


@pytest.mark.parametrize("variant", ["warp", "cta", "tma", "cluster", "generic"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_variant_parity(variant, dtype, M, N):
    wl = W.custom(M, N, dtype, seed=M * 131 + N, eps=1e-6, offset=float(N % 2 == 0 and M % 2))
    x, w = W.generate(wl)
    try:
        _plan(M, N, dtype, variant=variant)
    except B.RMSNormError as e:
        assert e.status == -8
        pytest.skip(f"{variant} does not take N={N}")
    for max_ctas, blocked in ((0, False), (2, False), (0, True), (3, True)):
        _run_and_check(x, w, dtype, wl.eps, wl.offset, variant=variant, max_ctas=max_ctas,
                       blocked=blocked, expect_variant=variant)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("N", [8, 64, 256, 512, 1000])
@pytest.mark.parametrize("D", [1, 2, 4])
def test_warp_lanes_per_row_and_ring_depth(G, N, D):
    if (N // 8 + G - 1) // G > 4:
        pytest.skip("more than 4 vectors per lane")
    wl = W.custom(203, N, "bf16", seed=G + N + D, offset=1.0)
    x, w = W.generate(wl)
    for max_ctas, blocked in ((0, False), (1, False), (3, True)):
        _run_and_check(x, w, "bf16", wl.eps, wl.offset, variant="warp", lanes_per_row=G,
                       stages=D, max_ctas=max_ctas, blocked=blocked, expect_variant="warp")


@pytest.mark.parametrize("variant,G", [("warp", 32), ("warp", 16), ("warp", 8), ("tma", 0),
                                       ("tma", 64)])
@pytest.mark.parametrize("M,N", [(37, 512), (257, 1000), (1000, 256), (130, 520), (64, 4096)])
@pytest.mark.parametrize("P", [1, 3, 15])
def test_l2_prefetch_parity(variant, G, M, N, P):
    # L2 prefetch of rows (warp) or chunks (TMA) ahead: a hint only, so the bits
    # must not change. Strict order and early loads, strided and blocked rows,
    # grids small enough that every team walks many rows, and in place.
    if G and (N // 8 + G - 1) // G > 4:
        pytest.skip("more than 4 vectors per lane")
    wl = W.custom(M, N, "bf16", seed=M + N + P + G, offset=float(P % 2))
    x, w = W.generate(wl)
    for max_ctas, blocked, early in ((0, False, False), (1, False, True), (3, True, False),
                                     (5, False, False)):
        _run_and_check(x, w, "bf16", wl.eps, wl.offset, variant=variant, lanes_per_row=G,
                       l2_prefetch=P, max_ctas=max_ctas, blocked=blocked, early_loads=early,
                       expect_variant=variant)
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, inplace=True, variant=variant,
                   lanes_per_row=G, l2_prefetch=P, max_ctas=2, expect_variant=variant)
    plan = _plan(M, N, "bf16", variant=variant, lanes_per_row=G, l2_prefetch=P)
    assert plan["l2_prefetch"] == P


@pytest.mark.parametrize("variant,G", [("warp", 32), ("warp", 8), ("warp", 4), ("tma", 0),
                                       ("tma", 64)])
@pytest.mark.parametrize("M,N", [(37, 512), (1000, 256), (130, 520), (64, 4096), (4099, 1000)])
@pytest.mark.parametrize("PW", [1, 4, 15])
def test_prewait_prefetch_parity(variant, G, M, N, PW):
    # Rows (warp) or chunks (TMA) asked into L2 before the wait for the previous
    # kernel: a hint only, so the bits must not change. Strict order and early
    # weights, strided and blocked rows, one CTA walking every row, in place,
    # and row strides wider than the row (one prefetch per row).
    if G and (N // 8 + G - 1) // G > 4:
        pytest.skip("more than 4 vectors per lane")
    wl = W.custom(M, N, "bf16", seed=M + N + PW + G, offset=float(PW % 2))
    x, w = W.generate(wl)
    for max_ctas, blocked, early_w in ((0, False, False), (1, False, True), (3, True, False),
                                       (5, False, True)):
        _run_and_check(x, w, "bf16", wl.eps, wl.offset, variant=variant, lanes_per_row=G,
                       prewait_prefetch=PW, max_ctas=max_ctas, blocked=blocked,
                       early_weights=early_w, expect_variant=variant)
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, inplace=True, variant=variant,
                   lanes_per_row=G, prewait_prefetch=PW, max_ctas=2, expect_variant=variant)
    # With early loads allowed, a positive count replaces the loads before the
    # wait (x is then read only after it).
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, variant=variant, lanes_per_row=G,
                   prewait_prefetch=PW, early_loads=True, expect_variant=variant)
    assert _plan(M, N, "bf16", variant=variant, lanes_per_row=G, prewait_prefetch=PW,
                 early_loads=True)["prewait_prefetch"] == PW
    plan = _plan(M, N, "bf16", variant=variant, lanes_per_row=G, prewait_prefetch=PW)
    assert plan["prewait_prefetch"] == PW
    ldx = ldy = N + 24
    _, _, xd, yd = _strided_case(x, w, "bf16", ldx, ldy)
    wd = W.to_torch(w, "bf16").cuda()
    rd = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
    o = B.make_options(variant=variant, lanes_per_row=G, prewait_prefetch=PW)
    rc = B.rmsnorm_fwd_strided(xd.data_ptr(), ldx, wd.data_ptr(), yd.data_ptr(), ldy,
                               rd.data_ptr(), M, N, wl.eps, wl.offset, B.BF16, o,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    torch.cuda.synchronize()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    yg = W.from_torch(yd).reshape(M, ldy)
    compare(yg[:, :N], rd.cpu().numpy(), yo, ro, "bf16", where=f"strided {M}x{N}")


@pytest.mark.parametrize("M,N,dtype,variant,per_sm,pw,P,early_pw", [
    (16384, 512, "bf16", "tma", 4, 1, 0, 1), (16384, 384, "bf16", "tma", 4, 1, 0, 1),
    (32768, 512, "bf16", "tma", 4, 2, 0, 2), (65536, 512, "bf16", "tma", 3, 3, 0, 3),
    (65536, 256, "bf16", "tma", 4, 2, 0, 2), (16384, 256, "bf16", "tma", 4, 1, 0, 0),
    (65536, 128, "bf16", "warp", 3, 3, 0, 0), (2048, 512, "bf16", "tma", 4, 1, 0, 0),
    (4096, 512, "bf16", "tma", 4, 1, 0, 0), (4096, 640, "bf16", "tma", 4, 1, 0, 1),
    (16384, 256, "fp32", "tma", 4, 1, 0, 1), (16384, 512, "fp32", "tma", 4, 2, 0, 2),
    (16384, 512, "fp16", "tma", 3, 2, 0, 2), (32768, 1000, "bf16", "tma", 3, 3, 0, 3),
    (16384, 8192, "bf16", "tma", 2, 3, 0, 0)])
def test_automatic_prewait_plan(M, N, dtype, variant, per_sm, pw, P, early_pw):
    # The planner's pre-wait prefetch under strict order: the kernel, its CTAs
    # per SM (four for the lean bf16 instances on batches up to 48 MB), the
    # rows or chunks it covers and the loop's own prefetch distance; with early
    # loads allowed, where it replaces the loads before the wait (early_pw > 0)
    # and where it does not; none without PDL or when the caller says -1.
    plan = _plan(M, N, dtype)
    assert plan["variant"] == variant and plan["ctas_per_sm"] == per_sm
    assert (plan["prewait_prefetch"], plan["l2_prefetch"]) == (pw, P)
    assert _plan(M, N, dtype, early_loads=True)["prewait_prefetch"] == early_pw
    assert _plan(M, N, dtype, pdl=False)["prewait_prefetch"] == 0
    assert _plan(M, N, dtype, prewait_prefetch=-1)["prewait_prefetch"] == 0
    assert _plan(M, N, dtype, early_loads=True, prewait_prefetch=-1)["prewait_prefetch"] == 0


def test_padded_shared_memory_holds_three_ctas_per_sm():
    # 512-byte bf16 rows in a 64 MB batch: the TMA instance's registers would
    # admit four CTAs per SM, so the planner pads the dynamic shared memory to
    # hold three; the kernel ignores the padding and every row must match.
    M, N = 131072, 256
    wl = W.custom(M, N, "bf16", seed=5)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "bf16")
    plan = _plan(M, N, "bf16", case)
    assert plan["variant"] == "tma" and plan["ctas_per_sm"] == 3
    assert plan["smem_bytes"] > 128 + 128 + plan["stages"] * plan["rows_per_stage"] * N * 2
    for early in (False, True):
        assert case.run(wl.eps, wl.offset, early_loads=early) == 0, B.rmsnorm_last_error()
        y, r = case.results()
        case.check_guards()
        yo, ro = oracle_threaded(x, w, wl.eps, wl.offset, "bf16")
        compare_blocked(y, r, yo, ro, "bf16", where=f"padded {M}x{N} early={early}")


@pytest.mark.parametrize("variant,N", [("warp", 512), ("warp", 256), ("tma", 1000), ("tma", 2048)])
@pytest.mark.parametrize("pw", [0, 1, 4])
def test_prewait_chain_keeps_stream_order(variant, N, pw):
    # A dependent chain at a size where the automatic plan prefetches before the
    # wait (each call reads the previous call's output): bit-identical to the
    # same calls separated by a device synchronize.
    M = 16384
    wl = W.custom(M, N, "bf16", seed=N + pw)
    x, w = W.generate(wl)
    w_dev = W.to_torch(w, "bf16").cuda()
    if pw:
        assert _plan(M, N, "bf16", variant=variant, prewait_prefetch=pw)["prewait_prefetch"] == pw
    else:
        assert _plan(M, N, "bf16", variant=variant)["prewait_prefetch"] > 0

    def chain(sync: bool):
        a = W.to_torch(x, "bf16").cuda()
        b = torch.empty_like(a)
        r = torch.empty(M, dtype=torch.float32, device="cuda")
        for _ in range(6):
            _raw_call(a, w_dev, b, r, M, N, 1e-6, 0.0, variant=variant, prewait_prefetch=pw)
            if sync:
                torch.cuda.synchronize()
            _raw_call(b, w_dev, a, r, M, N, 1e-6, 0.0, variant=variant, prewait_prefetch=pw)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return W.from_torch(a), r.cpu().numpy()

    ya, ra = chain(False)
    yb, rb = chain(True)
    assert np.array_equal(ya, yb) and np.array_equal(ra, rb)


@pytest.mark.parametrize("T", [64, 128, 256, 512, 1024])
@pytest.mark.parametrize("N", [512, 4096, 8192])
def test_cta_threads(T, N):
    if (N // 8 + T - 1) // T > 4:
        pytest.skip("more than 4 vectors per thread")
    wl = W.custom(41, N, "fp16", seed=T + N, x_std=30.0)
    x, w = W.generate(wl)
    for blocked in (False, True):
        _run_and_check(x, w, "fp16", wl.eps, wl.offset, variant="cta", lanes_per_row=T,
                       max_ctas=3, blocked=blocked, expect_variant="cta")


@pytest.mark.parametrize("team,rows,stages", [(16, 1, 1), (16, 7, 2), (32, 16, 3), (64, 5, 4),
                                              (128, 3, 2), (256, 1, 8), (512, 2, 2),
                                              (1024, 1, 3), (0, 0, 0)])
@pytest.mark.parametrize("N", [512, 1000, 4096, 8192])
def test_tma_team_rows_stages(team, rows, stages, N):
    wl = W.custom(77, N, "bf16", seed=team + rows + stages + N, outlier_p=0.01)
    x, w = W.generate(wl)
    try:
        _plan(77, N, "bf16", variant="tma", lanes_per_row=team, rows_per_stage=rows, stages=stages)
    except B.RMSNormError as e:
        assert e.status == -8
        pytest.skip("configuration not taken")
    for max_ctas, blocked in ((0, False), (1, False), (5, False), (0, True), (5, True)):
        _run_and_check(x, w, "bf16", wl.eps, wl.offset, variant="tma", lanes_per_row=team,
                       rows_per_stage=rows, stages=stages, max_ctas=max_ctas, blocked=blocked,
                       expect_variant="tma")


# ---------------------------------------------------------------- odd shapes, alignment

@pytest.mark.parametrize("N", [1, 2, 3, 7, 9, 31, 127, 1023, 1025, 4097, 8193])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_odd_n_takes_general_kernel(N, dtype):
    wl = W.custom(33, N, dtype, seed=N)
    x, w = W.generate(wl)
    for max_ctas in (0, 4):
        _run_and_check(x, w, dtype, wl.eps, wl.offset, max_ctas=max_ctas,
                       expect_variant="generic")


@pytest.mark.parametrize("x_shift,y_shift", [(1, 0), (0, 1), (3, 5), (4, 0)])
def test_misaligned_pointers(x_shift, y_shift):
    wl = W.custom(129, 512, "bf16", seed=x_shift * 10 + y_shift)
    x, w = W.generate(wl)
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, x_shift=x_shift, y_shift=y_shift,
                   expect_variant="generic")


@pytest.mark.parametrize("variant,N", [("warp", 512), ("warp", 1000), ("cta", 8192),
                                       ("tma", 512), ("tma", 8192), ("generic", 777),
                                       ("auto", 4096), ("cluster", 16384)])
def test_in_place(variant, N):
    wl = W.custom(300, N, "bf16", seed=N + 5)
    x, w = W.generate(wl)
    for blocked in (False, True):
        _run_and_check(x, w, "bf16", wl.eps, wl.offset, inplace=True, variant=variant, max_ctas=7,
                       blocked=blocked)


def test_zero_rows_and_eps_zero():
    # Row 0 all zeros with eps = 0: rstd = inf and y = NaN, as in IEEE fp32 and fp64.
    wl = W.custom(64, 512, "bf16", seed=3)
    x, w = W.generate(wl)
    x[0] = 0
    x[5] = 0
    for variant in ("warp", "cta", "tma", "cluster", "generic"):
        _run_and_check(x, w, "bf16", 0.0, 0.0, variant=variant)
    x[5, 7] = 0x3F80  # one 1.0
    _run_and_check(x, w, "bf16", 1e-5, 1.0)


def test_m_zero_launches_nothing():
    w = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_fwd(0, w.data_ptr(), 0, 0, 0, 512, 1e-6, 0.0, B.BF16, s) == 0


def test_torch_convenience_and_streams():
    wl = W.custom(1000, 1024, "fp16", seed=9)
    x, w = W.generate(wl)
    xt = W.to_torch(x, "fp16").cuda()
    wt = W.to_torch(w, "fp16").cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, r = B.fwd(xt, wt, eps=wl.eps, offset=wl.offset)
    s.synchronize()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp16")
    compare(W.from_torch(y), r.cpu().numpy(), yo, ro, "fp16")


# ---------------------------------------------------------------- past 2^31 elements

@pytest.mark.parametrize("variant,N", [("auto", 4096), ("tma", 4096), ("warp", 1024),
                                       ("generic", 1024)])
def test_more_than_2_31_elements(variant, N):
    block = 256
    M = (1 << 31) // N + 3 * block // 2  # ragged: the last block is cut in half
    wl = W.custom(block, N, "bf16", seed=N)
    xb, w = W.generate(wl)
    reps = (M + block - 1) // block
    x_dev = W.to_torch(xb, "bf16").cuda().repeat(reps, 1)[:M].contiguous()
    w_dev = W.to_torch(w, "bf16").cuda()
    y_dev = torch.empty_like(x_dev)
    r_dev = torch.empty(M, dtype=torch.float32, device="cuda")
    opts = B.make_options(variant=variant)
    rc = B.rmsnorm_fwd_ex(x_dev.data_ptr(), w_dev.data_ptr(), y_dev.data_ptr(), r_dev.data_ptr(),
                          M, N, wl.eps, 0.0, B.BF16, opts, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    rows = np.array([0, 1, block - 1, M // 2, (1 << 31) // N, (1 << 31) // N + 1, M - 2, M - 1])
    y = W.from_torch(y_dev[torch.from_numpy(rows).cuda()])
    r = r_dev.cpu().numpy()[rows]
    yo, ro = oracle.rmsnorm_fwd(xb, w, wl.eps, 0.0, "bf16")
    compare(y, r, yo[rows % block], ro[rows % block], "bf16", where=f"M={M}")
    del x_dev, y_dev
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- bounded waits

def test_tma_bounded_wait_reports_timeout_and_recovers():
    # A 1 ns wait bound makes the first stage's wait give up before its copy
    # lands: the kernel records the timeout, drains its own copies and exits.
    wl = W.custom(4096, 4096, "bf16", seed=11)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "bf16")
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_check_device_status(s) == 0
    assert case.run(wl.eps, wl.offset, variant="tma", wait_limit_ns=1) == 0
    assert B.rmsnorm_check_device_status(s) == -7
    assert B.rmsnorm_check_device_status(s) == 0  # the status word was cleared
    case.check_guards()
    # The context is still usable and a normal call is exact.
    assert case.run(wl.eps, wl.offset, variant="tma") == 0
    assert B.rmsnorm_check_device_status(s) == 0
    y, r = case.results()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    compare(y, r, yo, ro, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("N", [512, 1000, 4096, 8192])
@pytest.mark.parametrize("early", [False, True], ids=["strict", "early_loads"])
def test_tma_bulk_store(dtype, N, early):
    # y written into the shared-memory stage and copied out by cp.async.bulk:
    # same bits as per-thread stores, any grid, in place too.
    wl = W.custom(611, N, dtype, seed=N + 7, offset=float(early))
    x, w = W.generate(wl)
    for max_ctas in (0, 5):
        _run_and_check(x, w, dtype, wl.eps, wl.offset, variant="tma", bulk_store=True,
                       early_loads=early, max_ctas=max_ctas, expect_variant="tma")
    _run_and_check(x, w, dtype, wl.eps, wl.offset, inplace=True, variant="tma", bulk_store=True)
    a = DeviceCase(x, w, dtype)
    b = DeviceCase(x, w, dtype)
    assert a.run(wl.eps, wl.offset, variant="tma") == 0
    assert b.run(wl.eps, wl.offset, variant="tma", bulk_store=True) == 0
    ya, ra = a.results()
    yb, rb = b.results()
    assert np.array_equal(ya, yb) and np.array_equal(ra, rb)


@pytest.mark.parametrize("N", [1000, 8192])
def test_tma_bulk_store_chained_calls_and_timeout(N):
    # Each call reads the previous call's output: the bulk stores must have
    # completed before the next kernel reads y as its x.
    M = 3000
    wl = W.custom(M, N, "bf16", seed=N + 29)
    x, w = W.generate(wl)
    w_dev = W.to_torch(w, "bf16").cuda()

    def chain(sync: bool):
        a = W.to_torch(x, "bf16").cuda()
        b = torch.empty_like(a)
        r = torch.empty(M, dtype=torch.float32, device="cuda")
        for _ in range(8):
            _raw_call(a, w_dev, b, r, M, N, 1e-6, 0.0, variant="tma", bulk_store=True)
            if sync:
                torch.cuda.synchronize()
            _raw_call(b, w_dev, a, r, M, N, 1e-6, 0.0, variant="tma", bulk_store=True)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return W.from_torch(a), r.cpu().numpy()

    ya, ra = chain(False)
    yb, rb = chain(True)
    assert np.array_equal(ya, yb) and np.array_equal(ra, rb)
    # A wait that gives up: the CTA stops, waits for its bulk stores and loads,
    # and the next normal call is exact.
    case = DeviceCase(x, w, "bf16")
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_check_device_status(s) == 0
    assert case.run(wl.eps, wl.offset, variant="tma", bulk_store=True, wait_limit_ns=1) == 0
    assert B.rmsnorm_check_device_status(s) in (0, -7)
    case.check_guards()
    assert case.run(wl.eps, wl.offset, variant="tma", bulk_store=True) == 0
    assert B.rmsnorm_check_device_status(s) == 0
    y, r = case.results()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    compare(y, r, yo, ro, "bf16")


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 1000), ("cta", 16384),
                                       ("cluster", 65536), ("generic", 777)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_power_of_two_scale_invariance_on_gpu(variant, N, dtype):
    # eps = 0: y(2^k x) is y(x) within 1 ulp (the oracle's is exact), and
    # rstd(2^k x) is rstd(x) / 2^k within the rstd tolerance.
    M = 64 if N < 65536 else 8
    rng = np.random.default_rng(N)
    mag = rng.uniform(0.5, 2.0, (M, N)) * rng.choice([-1.0, 1.0], (M, N))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    x = W.from_torch(torch.from_numpy(mag).to(tdt))
    w = W.from_torch(torch.from_numpy(rng.uniform(0.5, 1.5, N)).to(tdt))
    outs = []
    for k in (0, 3, -2):
        xs = W.from_torch(W.to_torch(x, dtype).to(torch.float64).mul(2.0 ** k).to(tdt))
        case = DeviceCase(xs, w, dtype)
        assert case.run(0.0, 0.0, variant=variant) == 0, B.rmsnorm_last_error()
        y, r = case.results()
        outs.append((k, y, r))
    _, y0, r0 = outs[0]
    for k, y, r in outs[1:]:
        compare(y, r * 2.0 ** k, y0, r0.astype(np.float64), dtype, where=f"2^{k} x")


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 4096), ("cta", 16384),
                                       ("generic", 100)])
def test_gemma_identity_on_gpu(variant, N):
    # offset 1 with w = 0 equals offset 0 with w = 1: (offset + w) is 1 either way.
    wl = W.custom(128, N, "bf16", seed=N + 41)
    x, _ = W.generate(wl)
    zeros = W.from_torch(torch.zeros(N, dtype=torch.bfloat16))
    ones = W.from_torch(torch.ones(N, dtype=torch.bfloat16))
    a = DeviceCase(x, zeros, "bf16")
    b = DeviceCase(x, ones, "bf16")
    assert a.run(1e-6, 1.0, variant=variant) == 0
    assert b.run(1e-6, 0.0, variant=variant) == 0
    ya, ra = a.results()
    yb, rb = b.results()
    assert np.array_equal(ya, yb) and np.array_equal(ra, rb)
    yo, ro = oracle.rmsnorm_fwd(x, ones, 1e-6, 0.0, "bf16")
    compare(ya, ra, yo, ro, "bf16")


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 1000), ("cta", 16384),
                                       ("cluster", 65536), ("generic", 777)])
def test_nan_and_inf_propagate(variant, N):
    # Rows with a NaN give NaN rstd and y; rows with an Inf give rstd 0 and
    # y = +-0 except NaN at the Inf itself, as in the oracle (IEEE).
    M = 16
    wl = W.custom(M, N, "bf16", seed=N + 77)
    x, w = W.generate(wl)
    x[3, N // 2] = 0x7FC0   # NaN
    x[7, 1] = 0x7F80        # +Inf
    x[9, N - 1] = 0xFF80    # -Inf
    case = DeviceCase(x, w, "bf16")
    assert case.run(wl.eps, wl.offset, variant=variant) == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    assert np.isnan(r[3]) and r[7] == 0.0 and r[9] == 0.0
    compare(y, r, yo, ro, "bf16", where=f"nan/inf {variant}")


def test_results_are_deterministic():
    wl = W.WORKLOADS["rmsnorm_16384x512_bf16"]
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "bf16")
    outs = []
    for _ in range(3):
        assert case.run(wl.eps, wl.offset) == 0
        y, r = case.results()
        outs.append((y.copy(), r.copy()))
    assert all(np.array_equal(outs[0][0], o[0]) and np.array_equal(outs[0][1], o[1])
               for o in outs[1:])


# ---------------------------------------------------------------- stream order with PDL

def _raw_call(x, w, y, r, M, N, eps, offset, **opts):
    o = B.make_options(**opts) if opts else None
    rc = B.rmsnorm_fwd_ex(x.data_ptr(), w.data_ptr(), y.data_ptr(), r.data_ptr(), M, N, eps,
                          offset, B.BF16, o, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 1000), ("tma", 4096),
                                       ("cta", 8192), ("generic", 1000), ("cluster", 65536)])
@pytest.mark.parametrize("early_weights", [False, True], ids=["plain", "early_weights"])
def test_chained_calls_keep_stream_order(variant, N, early_weights):
    # Each call reads the previous call's output (ping-pong between two buffers),
    # launched back to back with programmatic dependent launch: the result must be
    # bit-identical to the same calls separated by a device synchronize. With
    # early weights the kernels read w before the previous call ends, but x
    # (the previous output) only after it.
    M = 3000
    wl = W.custom(M, N, "bf16", seed=N + 17)
    x, w = W.generate(wl)
    w_dev = W.to_torch(w, "bf16").cuda()

    def chain(sync: bool):
        a = W.to_torch(x, "bf16").cuda()
        b = torch.empty_like(a)
        r = torch.empty(M, dtype=torch.float32, device="cuda")
        for _ in range(12):
            _raw_call(a, w_dev, b, r, M, N, 1e-6, 0.0, variant=variant, early_weights=early_weights)
            if sync:
                torch.cuda.synchronize()
            _raw_call(b, w_dev, a, r, M, N, 1e-6, 0.0, variant=variant, early_weights=early_weights)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return W.from_torch(a), r.cpu().numpy()

    ya, ra = chain(False)
    yb, rb = chain(True)
    assert np.array_equal(ya, yb) and np.array_equal(ra, rb)


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 1000), ("tma", 8192), ("cta", 4096)])
def test_early_loads_on_independent_batches(variant, N):
    # With the early-loads promise (inputs not written by the previous kernel),
    # back-to-back calls on independent buffers still match the oracle.
    M = 2500
    wl = W.custom(M, N, "bf16", seed=N + 23, offset=1.0)
    x, w = W.generate(wl)
    xs = [W.to_torch(x, "bf16").cuda() for _ in range(4)]
    w_dev = W.to_torch(w, "bf16").cuda()
    ys = [torch.empty_like(xs[0]) for _ in range(4)]
    rs = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in range(4)]
    for rep in range(16):
        i = rep % 4
        _raw_call(xs[i], w_dev, ys[i], rs[i], M, N, wl.eps, wl.offset, variant=variant,
                  early_loads=True)
    torch.cuda.synchronize()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    for i in range(4):
        compare(W.from_torch(ys[i]), rs[i].cpu().numpy(), yo, ro, "bf16", where=f"buffer {i}")


# ---------------------------------------------------------------- long rows (cluster variant)

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M,N,C,S", [(37, 16384, 2, 2), (21, 65536, 0, 0), (19, 100000, 0, 0),
                                     (12, 131072, 4, 2), (9, 262144, 0, 1), (7, 65536, 16, 3),
                                     (64, 24576, 8, 4)])
def test_cluster_parity(dtype, M, N, C, S):
    wl = W.custom(M, N, dtype, seed=N + C, offset=float(C % 2), outlier_p=0.01)
    x, w = W.generate(wl)
    for max_ctas, early in ((0, False), (0, True), (C or 4, False)):
        _run_and_check(x, w, dtype, wl.eps, wl.offset, variant="cluster", cluster_size=C,
                       stages=S, max_ctas=max_ctas, early_loads=early, expect_variant="cluster")


def test_automatic_plan_takes_clusters_for_long_rows():
    wl = W.custom(40, 131072, "bf16", seed=5)
    x, w = W.generate(wl)
    p = _plan(40, 131072, "bf16")
    assert p["variant"] == "cluster" and p["cluster_size"] >= 2
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, expect_variant="cluster")
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, inplace=True, expect_variant="cluster")


def test_rows_beyond_cluster_reach_take_general_kernel():
    wl = W.custom(2, (1 << 21) + 8, "bf16", seed=6)
    x, w = W.generate(wl)
    _run_and_check(x, w, "bf16", wl.eps, wl.offset, expect_variant="generic")


def test_cluster_bounded_wait_reports_timeout_and_recovers():
    wl = W.custom(64, 65536, "bf16", seed=12)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "bf16")
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_check_device_status(s) == 0
    assert case.run(wl.eps, wl.offset, variant="cluster", wait_limit_ns=1) == 0
    assert B.rmsnorm_check_device_status(s) == -7
    assert B.rmsnorm_check_device_status(s) == 0
    case.check_guards()
    assert case.run(wl.eps, wl.offset, variant="cluster") == 0
    assert B.rmsnorm_check_device_status(s) == 0
    y, r = case.results()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    compare(y, r, yo, ro, "bf16")


# ---------------------------------------------------------------- strided rows, no rstd

def _strided_case(x, w, dtype, ldx, ldy, col0=0):
    """x rows inside a wider [M, ldx] buffer (canaries in the gaps), y into a [M, ldy] one."""
    M, N = x.shape
    nan = 0x7FC1 if dtype == "bf16" else 0x7E01
    xb = np.full((M, ldx + col0), nan, dtype=np.uint16)
    xb[:, col0:col0 + N] = x
    yb = np.full((M, ldy + col0), 0x5A5A, dtype=np.uint16)
    xd = W.to_torch(xb, dtype).cuda()
    yd = W.to_torch(yb, dtype).cuda()
    return xb, yb, xd, yd


@pytest.mark.parametrize("variant,N,ldx,ldy", [
    ("warp", 512, 640, 520), ("warp", 1000, 1000, 1024), ("cta", 8192, 8200, 8192),
    ("tma", 512, 520, 640), ("tma", 4096, 4104, 4096), ("tma", 8192, 16384, 8200),
    ("cluster", 65536, 65544, 65536), ("generic", 512, 513, 517), ("auto", 512, 513, 512),
    ("auto", 1000, 1008, 1000), ("auto", 8192, 8192, 8192)])
def test_strided_rows(variant, N, ldx, ldy):
    M = 300 if N < 65536 else 24
    wl = W.custom(M, N, "bf16", seed=N + ldx, offset=1.0)
    x, w = W.generate(wl)
    xb, yb, xd, yd = _strided_case(x, w, "bf16", ldx, ldy)
    wd = W.to_torch(w, "bf16").cuda()
    rd = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
    for early in (False, True):
        o = B.make_options(variant=variant, early_loads=early)
        rc = B.rmsnorm_fwd_strided(xd.data_ptr(), ldx, wd.data_ptr(), yd.data_ptr(), ldy,
                                   rd.data_ptr(), M, N, wl.eps, wl.offset, B.BF16, o,
                                   torch.cuda.current_stream().cuda_stream)
        assert rc == 0, B.rmsnorm_last_error()
        torch.cuda.synchronize()
        yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
        yg = W.from_torch(yd).reshape(M, ldy)
        compare(yg[:, :N], rd.cpu().numpy(), yo, ro, "bf16", where=f"{variant} ld {ldx}/{ldy}")
        assert np.all(yg[:, N:] == 0x5A5A), "y written between rows"
        assert np.array_equal(W.from_torch(xd).reshape(M, ldx), xb), "x changed"


def test_strided_in_place_and_torch_views():
    M, N, K = 257, 1024, 1536
    wl = W.custom(M, N, "fp16", seed=77, x_std=20.0)
    x, w = W.generate(wl)
    full = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    full[:, 256:256 + N] = W.to_torch(x, "fp16").cuda()
    view = full[:, 256:256 + N]          # rows of a wider tensor, 16-byte aligned
    wd = W.to_torch(w, "fp16").cuda()
    y, r = B.fwd(view, wd, eps=wl.eps, offset=wl.offset, y=view)   # in place, strided
    torch.cuda.synchronize()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp16")
    compare(W.from_torch(full[:, 256:256 + N].contiguous()), r.cpu().numpy(), yo, ro, "fp16")
    assert torch.count_nonzero(full[:, :256]) == 0 and torch.count_nonzero(full[:, 256 + N:]) == 0


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 1000), ("cta", 8192),
                                       ("cluster", 65536), ("generic", 777)])
def test_rstd_null_skips_the_store(variant, N):
    M = 200 if N < 65536 else 16
    wl = W.custom(M, N, "bf16", seed=N + 3)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "bf16")
    o = B.make_options(variant=variant)
    rc = B.rmsnorm_fwd_ex(case.x.data_ptr(), case.w.data_ptr(), case.y.data_ptr(), 0, M, N,
                          wl.eps, wl.offset, B.BF16, o, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    y, r = case.results()
    assert np.all(r == -12345.0)          # the rstd buffer was never written
    case.check_guards()
    yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    compare(y, ro, yo, ro, "bf16")
