"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on seeded inputs, run the oracle on the same bits, compare.

Tolerances (stated for the RMSNorm forward): y within 1 unit in the last place
of the output dtype for bf16/fp16 (for fp32 see ``compare_fp32``), rstd within
1e-5 relative of the oracle's fp64 value.
Derivation: the CUDA path computes in fp32; its sum of squares (at most a few
dozen sequential fp32 additions per thread, then a log-depth tree) and
rsqrt (<= 2 ulp) keep the relative error of rstd and of the unrounded y near
1e-6, far below half an ulp of bf16 (2^-9) or fp16 (2^-11), so the rounded y
can differ from the correctly rounded fp64 value by at most one step.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W

Y_ULP = 1
RSTD_REL = 1e-5
GUARD = 4096  # elements of canary on each side of every buffer
NAN_BITS = {"bf16": 0x7FC1, "fp16": 0x7E01, "fp32": 0x7FC00001}
SENTINEL = {"bf16": 0x5A5A, "fp16": 0x5A5A, "fp32": 0x5A5A5A5A}
RSTD_SENTINEL = -12345.0
DT = {"bf16": B.BF16, "fp16": B.FP16, "fp32": B.FP32}
TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
INT_DT = {"bf16": (torch.int16, np.int16), "fp16": (torch.int16, np.int16),
          "fp32": (torch.int32, np.int32)}
U32 = 2.0 ** -24  # unit roundoff of fp32


def ordinal(bits: np.ndarray) -> np.ndarray:
    """bf16/fp16 bit patterns -> integers in value order, +0 and -0 both 0."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def is_nan(bits: np.ndarray, dtype: str) -> np.ndarray:
    exp_mask, frac_mask = (0x7F80, 0x007F) if dtype == "bf16" else (0x7C00, 0x03FF)
    return ((bits & exp_mask) == exp_mask) & ((bits & frac_mask) != 0)


def compare(y_gpu, rstd_gpu, y_ref, rstd_ref, dtype, where=""):
    """Assert parity; returns (max ulp, max rstd rel err) for reporting."""
    y_gpu = np.asarray(y_gpu, dtype=np.uint16)
    y_ref = np.asarray(y_ref, dtype=np.uint16)
    assert y_gpu.shape == y_ref.shape, where
    ng, nr = is_nan(y_gpu, dtype), is_nan(y_ref, dtype)
    assert np.array_equal(ng, nr), f"{where}: NaN positions differ"
    d = np.abs(ordinal(y_gpu) - ordinal(y_ref))
    d[ng] = 0
    max_ulp = int(d.max()) if d.size else 0
    if max_ulp > Y_ULP:
        i = np.unravel_index(int(d.argmax()), d.shape)
        raise AssertionError(f"{where}: y off by {max_ulp} ulp at {i}: gpu {y_gpu[i]:#06x} "
                             f"oracle {y_ref[i]:#06x}")
    rg = np.asarray(rstd_gpu, dtype=np.float64)
    rr = np.asarray(rstd_ref, dtype=np.float64)
    same = (np.isinf(rg) & np.isinf(rr)) | (np.isnan(rg) & np.isnan(rr))
    with np.errstate(invalid="ignore"):
        rel = np.where(same, 0.0, np.abs(rg - rr) / np.where(rr == 0, 1, np.abs(rr)))
    rel = np.where(np.isnan(rel), np.inf, rel)  # NaN on one side only is a mismatch
    max_rel = float(rel.max()) if rel.size else 0.0
    if not max_rel <= RSTD_REL:
        i = int(np.nanargmax(rel))
        raise AssertionError(f"{where}: rstd rel err {max_rel:.3g} at row {i}: gpu {rg[i]!r} "
                             f"oracle {rr[i]!r}")
    return max_ulp, max_rel


def compare_fp32(y_gpu, rstd_gpu, y64, rstd_ref, where="", rstd_known=True):
    """fp32 parity. The CUDA path computes y = fl(fl(x * r) * fl(offset + w)),
    r its fp32 rstd; against the oracle's unrounded fp64 y this allows, per row,
    |y - y64| <= |y64| * (|r / r64 - 1| + 3u) (u = 2^-24), plus the smallest
    subnormal for products that underflow. rstd itself must stay within 1e-5.
    With ``rstd_known`` False (rstd not stored) the row factor is taken at its
    bound, 1e-5. Returns (max error in units of the bound, max rstd rel err,
    max ulp distance from the oracle's rounded y)."""
    y_gpu = np.asarray(y_gpu, dtype=np.uint32)
    g = y_gpu.view(np.float32).astype(np.float64)
    ng, nr = np.isnan(g), np.isnan(y64)
    assert np.array_equal(ng, nr), f"{where}: NaN positions differ"
    rr = np.asarray(rstd_ref, dtype=np.float64)
    if rstd_known:
        rg = np.asarray(rstd_gpu, dtype=np.float64)
        both_inf = np.isinf(rg) & np.isinf(rr)
        rel = np.where(both_inf, 0.0, np.abs(rg - rr) / np.where(rr == 0, 1, np.abs(rr)))
        max_rel = float(rel.max()) if rel.size else 0.0
        assert max_rel <= RSTD_REL, f"{where}: rstd rel err {max_rel:.3g}"
        with np.errstate(invalid="ignore"):
            rho = np.where(both_inf, 1.0, rg / np.where(rr == 0, 1, rr))
        row_term = np.abs(rho - 1.0)
    else:
        max_rel = float("nan")
        row_term = np.full(rr.shape, RSTD_REL)
    ok = ~nr
    bound = np.abs(y64) * (row_term[:, None] + 3.01 * U32 * (1 + row_term[:, None])) + 2.0 ** -149
    with np.errstate(invalid="ignore"):
        err = np.where(ok, np.abs(g - y64), 0.0)
    ratio = np.where(ok, err / bound, 0.0)
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(int(ratio.argmax()), ratio.shape)
        raise AssertionError(f"{where}: y off by {worst:.3g} of the bound at {i}: gpu {g[i]!r} "
                             f"oracle {y64[i]!r}")
    ref_bits = oracle.encode("fp32", np.where(ok, y64, 0.0))
    ulp = np.abs(ordinal32(y_gpu) - ordinal32(ref_bits))
    ulp[~ok] = 0
    return worst, max_rel, int(ulp.max()) if ulp.size else 0


def ordinal32(bits: np.ndarray) -> np.ndarray:
    """fp32 bit patterns -> integers in value order, +0 and -0 both 0."""
    b = np.asarray(bits, dtype=np.uint32).astype(np.int64)
    return np.where(b & 0x80000000, -(b & 0x7FFFFFFF), b)


class DeviceCase:
    """x, w, y, rstd on the GPU inside guarded buffers (canaries on both sides)."""

    def __init__(self, x_bits: np.ndarray, w_bits: np.ndarray, dtype: str, x_shift: int = 0,
                 y_shift: int = 0, inplace: bool = False, guard: int = GUARD):
        M, N = x_bits.shape
        self.M, self.N, self.dtype, self.guard = M, N, dtype, guard
        n = M * N
        tdt = TORCH_DT[dtype]
        ti, ni = INT_DT[dtype]
        nan = NAN_BITS[dtype]
        self.sentinel = SENTINEL[dtype]
        g = guard
        xb = torch.full((n + 2 * g + 8,), nan, dtype=ti)
        xb[g + x_shift: g + x_shift + n] = torch.from_numpy(x_bits.reshape(-1).view(ni))
        self.xbuf = xb.cuda().view(tdt)
        self.x = self.xbuf[g + x_shift: g + x_shift + n]
        wb = torch.full((N + 2 * g,), nan, dtype=ti)
        wb[g: g + N] = torch.from_numpy(w_bits.view(ni))
        self.wbuf = wb.cuda().view(tdt)
        self.w = self.wbuf[g: g + N]
        if inplace:
            self.ybuf, self.y = self.xbuf, self.x
        else:
            yb = torch.full((n + 2 * g + 8,), self.sentinel, dtype=ti)
            self.ybuf = yb.cuda().view(tdt)
            self.y = self.ybuf[g + y_shift: g + y_shift + n]
        self.y_shift = 0 if inplace else y_shift
        self.x_shift = x_shift
        self.inplace = inplace
        self.rbuf = torch.full((M + 2 * g,), RSTD_SENTINEL, dtype=torch.float32, device="cuda")
        self.rstd = self.rbuf[g: g + M]

    def run(self, eps: float, offset: float, stream: int | None = None, **opts) -> int:
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        o = B.make_options(**opts) if opts else None
        return B.rmsnorm_fwd_ex(self.x.data_ptr(), self.w.data_ptr(), self.y.data_ptr(),
                                self.rstd.data_ptr(), self.M, self.N, eps, offset,
                                DT[self.dtype], o, s)

    def results(self):
        torch.cuda.synchronize()
        y = W.from_torch(self.y).reshape(self.M, self.N)
        return y, self.rstd.cpu().numpy()

    def check_guards(self):
        torch.cuda.synchronize()
        g, n = self.guard, self.M * self.N
        nan = NAN_BITS[self.dtype]
        xb = W.from_torch(self.xbuf)
        lo, hi = g + self.x_shift, g + self.x_shift + n
        assert np.all(xb[:lo] == nan) and np.all(xb[hi:] == nan), "x guard changed"
        if not self.inplace:
            yb = W.from_torch(self.ybuf)
            lo, hi = g + self.y_shift, g + self.y_shift + n
            assert np.all(yb[:lo] == self.sentinel) and np.all(yb[hi:] == self.sentinel), \
                "y guard written"
        rb = self.rbuf.cpu().numpy()
        assert np.all(rb[:g] == RSTD_SENTINEL) and np.all(rb[g + self.M:] == RSTD_SENTINEL), \
            "rstd guard written"
        wb = W.from_torch(self.wbuf)
        assert np.all(wb[:g] == nan) and np.all(wb[g + self.N:] == nan), "w guard changed"


def oracle_rows(x_bits, w_bits, eps, offset, dtype, rows=None, want_y64=False):
    """Oracle on all rows, or on the listed row indices (gathered)."""
    if rows is None:
        return oracle.rmsnorm_fwd(x_bits, w_bits, eps, offset, dtype, want_y64=want_y64)
    xs = np.ascontiguousarray(x_bits[rows])
    return oracle.rmsnorm_fwd(xs, w_bits, eps, offset, dtype, want_y64=want_y64)


def oracle_threaded(x_bits, w_bits, eps, offset, dtype, threads: int | None = None):
    """The oracle on every row, the rows split into contiguous blocks over host
    threads (ctypes releases the GIL during each C call). Same result as
    ``oracle.rmsnorm_fwd`` on the whole array: each row is computed alone."""
    import os
    import threading
    x_bits = np.ascontiguousarray(x_bits, dtype=oracle.bits_dtype(dtype))
    w_bits = np.ascontiguousarray(w_bits, dtype=oracle.bits_dtype(dtype))
    M, N = x_bits.shape
    y = np.empty((M, N), dtype=oracle.bits_dtype(dtype))
    r = np.empty(M, dtype=np.float64)
    n = max(1, min(threads or os.cpu_count() or 1, M))
    bounds = [M * i // n for i in range(n + 1)]
    oracle.lib()
    ts = [threading.Thread(target=oracle.rmsnorm_fwd_into,
                           args=(x_bits, w_bits, y, r, eps, offset, dtype, bounds[i], bounds[i + 1]))
          for i in range(n) if bounds[i + 1] > bounds[i]]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return y, r


def compare_blocked(y_gpu, rstd_gpu, y_ref, rstd_ref, dtype, where="", block_elems=1 << 24):
    """``compare`` over blocks of rows (bounded temporaries for GiB-sized
    outputs). Returns (max ulp, max rstd rel err, {ulp distance: count})."""
    M, N = y_ref.shape
    rows = max(1, block_elems // N)
    max_ulp, max_rel, hist = 0, 0.0, {}
    for r0 in range(0, M, rows):
        r1 = min(M, r0 + rows)
        u, e = compare(y_gpu[r0:r1], rstd_gpu[r0:r1], y_ref[r0:r1], rstd_ref[r0:r1], dtype,
                       where=f"{where} rows {r0}..{r1 - 1}")
        d = np.abs(ordinal(np.asarray(y_gpu[r0:r1], dtype=np.uint16))
                   - ordinal(np.asarray(y_ref[r0:r1], dtype=np.uint16)))
        d[is_nan(np.asarray(y_gpu[r0:r1], dtype=np.uint16), dtype)] = 0
        for k, c in enumerate(np.bincount(d.ravel())):
            if c:
                hist[k] = hist.get(k, 0) + int(c)
        max_ulp, max_rel = max(max_ulp, u), max(max_rel, e)
    return max_ulp, max_rel, hist


def sample_rows(M: int, k: int, seed: int = 0) -> np.ndarray:
    """First, last and k random rows (sorted, unique)."""
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(M, size=min(k, M), replace=False).tolist())
    idx.update({0, M - 1, M // 2})
    return np.array(sorted(idx), dtype=np.int64)
