"""GPU tests of rmsnorm_fwd_host: x, y and rstd in host memory, moved through
the device ring in chunks of rows, against the fp64 oracle (same tolerances as
the device path: y within 1 ulp for bf16/fp16, the fp32 bound of
``parity_util.compare_fp32``; rstd within 1e-5) and bit for bit against the
device-resident call on the same inputs (the per-row arithmetic does not
depend on how rows are grouped into launches).
"""
from __future__ import annotations

import pytest
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W
from parity_util import compare, compare_fp32

pytestmark = pytest.mark.gpu


def _oracle_check(x, w, y_bits, rstd, wl, where=""):
    if wl.dtype == "fp32":
        _, ro, y64 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "fp32", want_y64=True)
        compare_fp32(y_bits, rstd, y64, ro, where=where, rstd_known=rstd is not None)
    else:
        yo, ro = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, wl.dtype)
        compare(y_bits, ro if rstd is None else rstd, yo, ro, wl.dtype, where=where)


def _device_reference(xt, wd, wl):
    y, r = B.fwd(xt.cuda(), wd, eps=wl.eps, offset=wl.offset)
    torch.cuda.synchronize()
    return y.cpu(), r.cpu()


CASES = [(16384, 512, "bf16", 0), (1000, 1000, "bf16", 7), (777, 4096, "fp16", 100),
         (5, 8192, "fp32", 2), (3000, 777, "bf16", 1000), (1, 8, "bf16", 0),
         (4099, 2048, "fp32", 0), (64, 65536, "bf16", 5), (300, 12, "fp16", 299)]


@pytest.mark.parametrize("M,N,dtype,chunk", CASES)
def test_host_path_matches_oracle_and_device_path(M, N, dtype, chunk):
    wl = W.custom(M, N, dtype, seed=M + N + chunk, offset=float(N % 2 == 0))
    x, w = W.generate(wl)
    xt = W.to_torch(x, dtype).pin_memory()
    wd = W.to_torch(w, dtype).cuda()
    y, r = B.fwd_host(xt, wd, eps=wl.eps, offset=wl.offset, chunk_rows=chunk)
    torch.cuda.synchronize()
    _oracle_check(x, w, W.from_torch(y), r.numpy(), wl, where=f"{M}x{N} {dtype} chunk {chunk}")
    yd, rd = _device_reference(xt, wd, wl)
    assert torch.equal(y.view(torch.int16 if dtype != "fp32" else torch.int32),
                       yd.view(torch.int16 if dtype != "fp32" else torch.int32))
    assert torch.equal(r, rd)


def test_in_place_rstd_null_and_pageable_memory():
    wl = W.custom(2500, 1024, "bf16", seed=41, offset=1.0)
    x, w = W.generate(wl)
    wd = W.to_torch(w, "bf16").cuda()
    # in place on pinned memory, rstd not stored
    buf = W.to_torch(x, "bf16").pin_memory()
    y, r = B.fwd_host(buf, wd, eps=wl.eps, offset=wl.offset, y=buf, rstd=False, chunk_rows=333)
    torch.cuda.synchronize()
    assert r is None and y.data_ptr() == buf.data_ptr()
    _oracle_check(x, w, W.from_torch(buf), None, wl, where="in place")
    # pageable (not pinned) host memory: correct, just without overlap
    xp = W.to_torch(x, "bf16").clone()
    yp = torch.empty_like(xp)
    rp = torch.empty(2500, dtype=torch.float32)
    B.fwd_host(xp, wd, eps=wl.eps, offset=wl.offset, y=yp, rstd=rp, chunk_rows=500)
    torch.cuda.synchronize()
    assert torch.equal(yp.view(torch.int16), buf.view(torch.int16))
    _oracle_check(x, w, W.from_torch(yp), rp.numpy(), wl, where="pageable")


def test_back_to_back_calls_reuse_the_workspace_on_a_side_stream():
    # Several calls queued without synchronising, one workspace, a non-default
    # stream: each call's chunks must wait for the previous call's copy-out
    # before reusing a slot, and each result must be that call's own.
    N, M = 512, 6000
    wd = None
    calls = []
    s = torch.cuda.Stream()
    need = B.rmsnorm_fwd_host_workspace_size(M, N, B.BF16, 1000)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for k in range(5):
        wl = W.custom(M, N, "bf16", seed=100 + k)
        x, w = W.generate(wl)
        if wd is None:
            wd = W.to_torch(w, "bf16").cuda()
            w0 = w
        xt = W.to_torch(x, "bf16").pin_memory()
        y, r = B.fwd_host(xt, wd, eps=wl.eps, offset=wl.offset, chunk_rows=1000, workspace=ws,
                          stream=s)
        calls.append((x, y, r, wl))
    s.synchronize()
    for x, y, r, wl in calls:
        _oracle_check(x, w0, W.from_torch(y), r.numpy(), wl, where=f"seed {wl.seed}")


def test_work_after_the_call_on_the_stream_sees_the_results():
    # Stream order: a device->host copy queued after the call on the same stream
    # runs only after the host-side y is complete, so copying y back to the GPU
    # and comparing there sees the final values.
    wl = W.custom(8192, 1024, "fp16", seed=7)
    x, w = W.generate(wl)
    xt = W.to_torch(x, "fp16").pin_memory()
    wd = W.to_torch(w, "fp16").cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, r = B.fwd_host(xt, wd, eps=wl.eps, offset=wl.offset, chunk_rows=512, stream=s)
        back = y.to("cuda", non_blocking=True)
        yd, _ = B.fwd(xt.to("cuda", non_blocking=True), wd, eps=wl.eps, offset=wl.offset)
        same = torch.equal(back.view(torch.int16), yd.view(torch.int16))
    s.synchronize()
    assert same


def test_forced_variant_that_cannot_run_fails_before_queuing():
    wl = W.custom(100, 777, "bf16", seed=9)
    x, w = W.generate(wl)
    xt = W.to_torch(x, "bf16").pin_memory()
    y = torch.full_like(xt, 3.0).pin_memory()
    wd = W.to_torch(w, "bf16").cuda()
    with pytest.raises(B.RMSNormError) as e:
        B.fwd_host(xt, wd, y=y, variant="warp")          # N % 8 != 0: no vector kernel
    assert e.value.status == -8
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


# ---------------------------------------------------------------- host-direct mode

@pytest.mark.parametrize("M,N,dtype", [(16384, 512, "bf16"), (777, 4096, "fp16"), (300, 1000, "fp32"),
                                       (50, 20000, "bf16"), (33, 777, "bf16"), (8, 100000, "bf16")])
def test_host_direct_matches_oracle_and_device_path(M, N, dtype):
    wl = W.custom(M, N, dtype, seed=M + 3 * N, offset=1.0)
    x, w = W.generate(wl)
    xt = W.to_torch(x, dtype).pin_memory()
    wd = W.to_torch(w, dtype).cuda()
    y, r = B.fwd_host(xt, wd, eps=wl.eps, offset=wl.offset, host_direct=True)
    torch.cuda.synchronize()
    _oracle_check(x, w, W.from_torch(y), r.numpy(), wl, where=f"direct {M}x{N} {dtype}")
    if N * W.ELEM_BYTES[dtype] <= 65536:
        # Same bits as the device call: host-direct runs the device plan's
        # kernel, or for a TMA plan the plain-load kernel with the same team and
        # vectors per thread (the same sum order). Rows over 64 KB take the
        # cluster kernel on the device and the general kernel here, whose sums
        # associate differently: oracle parity only.
        yd, rd = _device_reference(xt, wd, wl)
        iv = torch.int32 if dtype == "fp32" else torch.int16
        assert torch.equal(y.view(iv), yd.view(iv)) and torch.equal(r, rd)


def test_host_direct_in_place_rstd_null_and_refusals():
    wl = W.custom(4000, 1024, "bf16", seed=61)
    x, w = W.generate(wl)
    wd = W.to_torch(w, "bf16").cuda()
    buf = W.to_torch(x, "bf16").pin_memory()
    B.fwd_host(buf, wd, eps=wl.eps, y=buf, rstd=False, host_direct=True)
    torch.cuda.synchronize()
    _oracle_check(x, w, W.from_torch(buf), None, wl, where="direct in place")
    # pageable memory cannot be reached by the kernel through a device address
    xp = W.to_torch(x, "bf16").clone()
    with pytest.raises(B.RMSNormError) as e:
        B.fwd_host(xp, wd, y=torch.empty_like(xp), rstd=torch.empty(4000), host_direct=True)
    assert e.value.status == -8
    # bulk-copy kernels are refused in this mode
    with pytest.raises(B.RMSNormError) as e:
        B.fwd_host(W.to_torch(x, "bf16").pin_memory(), wd, host_direct=True, variant="tma")
    assert e.value.status == -8
