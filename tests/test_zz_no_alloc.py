"""rmsnorm_bwd_noalloc, the backward for callers that cannot allocate device
memory when they call it (a plugin inside a host framework that owns every
device allocation, or a real-time path whose memory plan is fixed at
start-up). It keeps the dw partials in scratch built into the library instead
of a caller workspace. Its results must match the workspace entry point's,
rmsnorm_bwd, within the backward tests' tolerance, on two calls in a row.

This file is collected last on purpose, and it needs nothing from the tests
before it: it passes alone in a fresh process and after the full suite.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TAU = 1e-5  # the backward tests' relative bound on an fp32 dw sum (see test_bwd_gpu.py)
DT = {"bf16": B.BF16, "fp16": B.FP16, "fp32": B.FP32}


def _inputs(M, N, dtype, seed):
    x, w = W.generate(W.custom(M, N, dtype, seed=seed))
    dy, _ = W.generate(W.custom(M, N, dtype, seed=seed + 500))
    xd, wd, gd = (W.to_torch(a, dtype).cuda() for a in (x, w, dy))
    # rstd as a forward would keep it: 1/sqrt(mean(x^2) + eps), fp32.
    rd = torch.rsqrt(xd.double().pow(2).mean(-1) + 1e-6).float()
    return xd, wd, gd, rd


def _with_workspace(xd, wd, rd, gd, offset, dtype):
    M, N = xd.shape
    dx = torch.empty_like(xd)
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    nbytes = B.rmsnorm_bwd_workspace_size(M, N, DT[dtype])
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    rc = B.rmsnorm_bwd(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), gd.data_ptr(), dx.data_ptr(),
                       dw.data_ptr(), M, N, offset, DT[dtype], ws.data_ptr(), ws.numel() * 4,
                       None, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    return dx, dw


def _no_alloc(xd, wd, rd, gd, offset, dtype):
    M, N = xd.shape
    dx = torch.empty_like(xd)
    dw = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    rc = B.rmsnorm_bwd_noalloc(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), gd.data_ptr(),
                               dx.data_ptr(), dw.data_ptr(), M, N, offset, DT[dtype], None,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.rmsnorm_last_error()
    return dx, dw


def _ordinal(t):
    b = W.from_torch(t).astype(np.int64)
    sign = 0x80000000 if t.dtype == torch.float32 else 0x8000
    return np.where(b & sign, -(b & (sign - 1)), b)


@pytest.mark.parametrize("M,N,dtype", [(20000, 8192, "bf16"), (777, 512, "fp16"),
                                       (50, 777, "bf16"), (3, 16384, "fp16"), (4000, 1000, "fp32"),
                                       (40, 100000, "bf16")])
def test_no_alloc_backward_matches_the_workspace_backward(M, N, dtype):
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        xd, wd, gd, rd = _inputs(M, N, dtype, seed + N)
        offset = float(call)
        ref_dx, ref_dw = _with_workspace(xd, wd, rd, gd, offset, dtype)
        dx, dw = _no_alloc(xd, wd, rd, gd, offset, dtype)
        torch.cuda.synchronize()
        # dx does not depend on how rows are dealt to CTAs: at most 1 ulp.
        assert np.abs(_ordinal(dx) - _ordinal(ref_dx)).max() <= 1
        # dw sums the same terms in another grouping (the grid may be capped):
        # each result lies within TAU * sum|dy x r| of the exact sum.
        bound = 2 * TAU * (gd.double() * xd.double() * rd.double()[:, None]).abs().sum(0) + 1e-30
        assert torch.all((dw.double() - ref_dw.double()).abs() <= bound), f"call {call}"
        assert torch.isfinite(dw).all()


def test_no_alloc_rejects_bad_arguments_on_the_host():
    # Argument errors come back before any device work (null dw, unknown dtype).
    wd = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert B.rmsnorm_bwd_noalloc(0, wd.data_ptr(), 0, 0, 0, 0, 0, 64, 0.0, B.BF16, None, s) == -1
    assert B.rmsnorm_bwd_noalloc(0, wd.data_ptr(), 0, 0, 0, 0, 0, 64, 0.0, 7, None, s) == -3


def test_no_alloc_refuses_rows_longer_than_its_scratch():
    # One partial row of N fp32 values must fit the built-in 8 MiB scratch
    # (2^21 values): a longer row is refused before any launch, dw untouched.
    N = (1 << 21) + 8
    xd = torch.zeros((1, N), dtype=torch.bfloat16, device="cuda")
    gd, dxd = torch.zeros_like(xd), torch.zeros_like(xd)
    wd = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    rd = torch.ones(1, dtype=torch.float32, device="cuda")
    dwd = torch.full((N,), 5.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = B.rmsnorm_bwd_noalloc(xd.data_ptr(), wd.data_ptr(), rd.data_ptr(), gd.data_ptr(),
                               dxd.data_ptr(), dwd.data_ptr(), 1, N, 0.0, B.BF16, None, s)
    assert rc == -11 and "scratch" in B.rmsnorm_last_error()
    torch.cuda.synchronize()
    assert torch.all(dwd == 5.0)


@pytest.mark.parametrize("dtype,N", [("bf16", 512), ("fp16", 1000), ("fp32", 8192)])
def test_no_alloc_with_no_rows_writes_zero_dw(dtype, N):
    # M = 0: no row kernel runs and nothing touches the scratch; the reduction
    # over zero partial rows must still write dw = 0 (NaN before the call),
    # on two calls in a row. x, dy, dx and rstd may be NULL when there are no rows.
    wd = W.to_torch(W.generate(W.custom(1, N, dtype, seed=N))[1], dtype).cuda()
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dw = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        rc = B.rmsnorm_bwd_noalloc(0, wd.data_ptr(), 0, 0, 0, dw.data_ptr(), 0, N, 1.0, DT[dtype],
                                   None, s)
        assert rc == 0, B.rmsnorm_last_error()
        torch.cuda.synchronize()
        assert torch.all(dw == 0.0)
