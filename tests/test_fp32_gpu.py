"""GPU parity for fp32 activations (x, w, y in fp32) through the C ABI, against
the oracle's fp64 forward on the same seeded inputs.

Tolerance (derived in ``parity_util.compare_fp32``): the CUDA path's y is the
fp32 product fl(fl(x * r) * fl(offset + w)) with r its own fp32 rstd, so per
row |y - y64| <= |y64| (|r / r64 - 1| + 3u), u = 2^-24; rstd within 1e-5
relative of the oracle's fp64 value, as for the 16-bit formats.

Covers every kernel variant on shapes spanning several tiles with ragged
tails, forced small grids, the automatic plan on full-size fp32 versions of
the benchmark shapes in both launch modes, rows that are not whole 16-byte
vectors and 4-byte-misaligned pointers (general kernel), in-place calls,
strided rows, rstd = NULL, zero rows and canaries around every buffer.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W
from parity_util import DeviceCase, compare_fp32, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu


def _check(x, w, eps, offset, rows=None, x_shift=0, y_shift=0, inplace=False, runs=1,
           expect_variant=None, **opts):
    M, N = x.shape
    case = DeviceCase(x, w, "fp32", x_shift=x_shift, y_shift=y_shift, inplace=inplace)
    if expect_variant is not None:
        plan = B.rmsnorm_plan_info(M, N, B.FP32, case.x.data_ptr(), case.w.data_ptr(),
                                   case.y.data_ptr(), B.make_options(**opts) if opts else None)
        assert plan["variant"] == expect_variant, plan
    for _ in range(runs):
        rc = case.run(eps, offset, **opts)
        assert rc == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    _, ro, y64 = oracle_rows(x, w, eps, offset, "fp32", rows, want_y64=True)
    if rows is not None:
        y, r = y[rows], r[rows]
    return compare_fp32(y, r, y64, ro, where=f"fp32 {x.shape} {opts}")


SHAPES = [(1, 4), (37, 512), (300, 1000), (64, 2048), (33, 4096), (17, 8192), (9, 16384),
          (5, 20000), (130, 516), (3, 65536)]


@pytest.mark.parametrize("variant", ["warp", "cta", "tma", "cluster", "generic"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_variant_parity(variant, M, N):
    wl = W.custom(M, N, "fp32", seed=M * 17 + N, offset=float((M + N) % 2))
    x, w = W.generate(wl)
    try:
        B.rmsnorm_plan_info(M, N, B.FP32, opts=B.make_options(variant=variant))
    except B.RMSNormError as e:
        assert e.status == -8
        pytest.skip("variant does not take this shape")
    for max_ctas in (0, 3):
        _check(x, w, wl.eps, wl.offset, variant=variant, max_ctas=max_ctas)


FULL = [
    W.Workload("fp32_16384x512", 16384, 512, dtype="fp32"),
    W.Workload("fp32_32768x1000_gemma", 32768, 1000, dtype="fp32", w_kind="normal", w_a=0.0,
               w_b=0.1, offset=1.0),
    W.Workload("fp32_4096x8192_heavytail", 4096, 8192, dtype="fp32", outlier_p=0.01,
               outlier_std=100.0, eps=1e-5),
    W.Workload("fp32_16384x4096_wide", 16384, 4096, dtype="fp32", x_std=64.0),
]


@pytest.mark.parametrize("early", [False, True], ids=["strict", "early_loads"])
@pytest.mark.parametrize("wl", FULL, ids=lambda w: w.name)
def test_full_size_automatic_launch(wl, early):
    x, w = W.generate(wl)
    rows = None if wl.M * wl.N <= (1 << 23) else sample_rows(wl.M, 160, seed=2)
    _check(x, w, wl.eps, wl.offset, rows=rows, runs=2 if early else 1, early_loads=early)


@pytest.mark.parametrize("N,variant,without_prewait", [
    (64, "warp", "warp"), (256, "tma", "warp"), (384, "tma", "warp"), (512, "tma", "tma"),
    (4096, "tma", "tma"), (8192, "cta", "cta"), (16384, "cta", "cta"),
    (32768, "cluster", "cluster")])
def test_planner_switches_at_row_bytes(N, variant, without_prewait):
    # The planner's limits are row bytes: an fp32 row switches kernels at half
    # the column count of a bf16 row. Under strict order rows over 256 bytes
    # take the TMA kernel with the pre-wait prefetch; without it (-1) the warp
    # kernel keeps rows of up to 1.5 KB.
    wl = W.custom(64, N, "fp32", seed=N)
    x, w = W.generate(wl)
    _check(x, w, wl.eps, wl.offset, expect_variant=variant)
    _check(x, w, wl.eps, wl.offset, expect_variant=without_prewait, prewait_prefetch=-1)


@pytest.mark.parametrize("N", [1, 2, 3, 5, 7, 9, 31, 127, 1023, 1025, 4097])
def test_rows_not_whole_vectors_take_general_kernel(N):
    wl = W.custom(33, N, "fp32", seed=N + 300)
    x, w = W.generate(wl)
    for max_ctas in (0, 5):
        _check(x, w, wl.eps, wl.offset, expect_variant="generic", max_ctas=max_ctas)


@pytest.mark.parametrize("x_shift,y_shift", [(1, 0), (0, 1), (3, 2), (4, 0)])
def test_misaligned_pointers(x_shift, y_shift):
    wl = W.custom(129, 512, "fp32", seed=x_shift * 10 + y_shift + 500)
    x, w = W.generate(wl)
    _check(x, w, wl.eps, wl.offset, x_shift=x_shift, y_shift=y_shift)


@pytest.mark.parametrize("variant,N", [("warp", 256), ("tma", 1000), ("cta", 8192),
                                       ("cluster", 32768), ("generic", 777)])
def test_in_place(variant, N):
    M = 300 if N < 32768 else 24
    wl = W.custom(M, N, "fp32", seed=N + 600)
    x, w = W.generate(wl)
    _check(x, w, wl.eps, wl.offset, inplace=True, variant=variant)


@pytest.mark.parametrize("variant,N,ldx,ldy", [("auto", 512, 512 + 4, 512 + 8),
                                               ("tma", 1000, 1024, 1000),
                                               ("cta", 8192, 8192 + 12, 8192 + 4),
                                               ("generic", 510, 515, 511)])
def test_strided_rows(variant, N, ldx, ldy):
    M = 200
    wl = W.custom(M, N, "fp32", seed=N + ldx)
    x, w = W.generate(wl)
    xfull = np.full((M, ldx), 0x7FC00001, dtype=np.uint32)
    xfull[:, :N] = x
    xd = torch.from_numpy(xfull.view(np.int32)).cuda().view(torch.float32)
    yd = torch.full((M, ldy), 0x5A5A5A5A, dtype=torch.int32, device="cuda").view(torch.float32)
    wd = W.to_torch(w, "fp32").cuda()
    rd = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
    rc = B.rmsnorm_fwd_strided(xd.data_ptr(), ldx, wd.data_ptr(), yd.data_ptr(), ldy,
                               rd.data_ptr(), M, N, wl.eps, wl.offset, B.FP32,
                               B.make_options(variant=variant),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    torch.cuda.synchronize()
    _, ro, y64 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp32", want_y64=True)
    yg = W.from_torch(yd).reshape(M, ldy)
    compare_fp32(yg[:, :N], rd.cpu().numpy(), y64, ro, where=f"strided {variant}")
    assert np.all(yg[:, N:] == 0x5A5A5A5A), "y written between rows"


@pytest.mark.parametrize("variant,N", [("warp", 512), ("tma", 2048), ("generic", 99)])
def test_rstd_null_and_torch_convenience(variant, N):
    wl = W.custom(150, N, "fp32", seed=N + 700, offset=1.0)
    x, w = W.generate(wl)
    xd, wd = W.to_torch(x, "fp32").cuda(), W.to_torch(w, "fp32").cuda()
    y, r = B.fwd(xd, wd, eps=wl.eps, offset=wl.offset, rstd=False, variant=variant)
    assert r is None
    torch.cuda.synchronize()
    _, ro, y64 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp32", want_y64=True)
    compare_fp32(W.from_torch(y), None, y64, ro, rstd_known=False)
    y2, r2 = B.fwd(xd, wd, eps=wl.eps, offset=wl.offset, variant=variant)
    torch.cuda.synchronize()
    compare_fp32(W.from_torch(y2), r2.cpu().numpy(), y64, ro)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("N", [256, 1000, 4096])
def test_tma_bulk_store(N):
    wl = W.custom(700, N, "fp32", seed=N + 900)
    x, w = W.generate(wl)
    for early in (False, True):
        _check(x, w, wl.eps, wl.offset, variant="tma", bulk_store=True, early_loads=early,
               runs=2 if early else 1)
    _check(x, w, wl.eps, wl.offset, inplace=True, variant="tma", bulk_store=True)


def test_zero_rows_and_eps_zero_give_nan():
    wl = W.custom(64, 512, "fp32", seed=800)
    x, w = W.generate(wl)
    x[5] = 0
    x[40] = 0
    worst, _, _ = _check(x, w, 0.0, 0.0)
    assert worst <= 1.0


def test_results_are_deterministic():
    wl = W.custom(4096, 1024, "fp32", seed=900)
    x, w = W.generate(wl)
    case = DeviceCase(x, w, "fp32")
    outs = []
    for _ in range(3):
        assert case.run(wl.eps, wl.offset) == 0
        outs.append(case.results())
    assert all(np.array_equal(outs[0][0], o[0]) and np.array_equal(outs[0][1], o[1]) for o in outs)
