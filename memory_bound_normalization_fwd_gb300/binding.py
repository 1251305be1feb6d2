"""Thin Python binding of the C ABI in include/rmsnorm.h (ctypes).

Argument marshalling only: every step of the RMSNorm forward runs in the CUDA
library. The raw functions keep the C names and take integer device
addresses; ``fwd`` is a convenience over torch tensors (torch supplies device
memory and the current stream, nothing else). There is no fallback: if the
library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

BF16, FP16, FP32 = 0, 1, 2
VARIANTS = {"auto": 0, "warp": 1, "cta": 2, "tma": 3, "generic": 4, "cluster": 5}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}
STATUS = {
    0: "RMSNORM_OK", -1: "RMSNORM_ERR_NULL", -2: "RMSNORM_ERR_SHAPE", -3: "RMSNORM_ERR_DTYPE",
    -4: "RMSNORM_ERR_SCALAR", -5: "RMSNORM_ERR_OVERLAP", -6: "RMSNORM_ERR_CUDA",
    -7: "RMSNORM_ERR_DEVICE_TIMEOUT", -8: "RMSNORM_ERR_UNSUPPORTED", -9: "RMSNORM_ERR_OPTIONS",
    -10: "RMSNORM_ERR_ALIGN", -11: "RMSNORM_ERR_WORKSPACE",
}
# Every function include/rmsnorm.h declares.
EXPORTS = ("rmsnorm_fwd", "rmsnorm_fwd_ex", "rmsnorm_fwd_strided", "rmsnorm_fwd_host",
           "rmsnorm_fwd_host_workspace_size", "rmsnorm_bwd", "rmsnorm_bwd_noalloc",
           "rmsnorm_bwd_workspace_size", "rmsnorm_plan_info", "rmsnorm_bwd_plan_info",
           "rmsnorm_check_device_status",
           "rmsnorm_strerror", "rmsnorm_last_error", "rmsnorm_version")


class RMSNormError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("lanes_per_row", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("rows_per_stage", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("l2_prefetch", ctypes.c_int32),
                ("prewait_prefetch", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "variant", "threads", "grid", "lanes_per_row", "vecs_per_lane", "rows_per_stage",
        "stages", "smem_bytes", "ctas_per_sm", "sm_count", "cluster_size", "l2_prefetch",
        "prewait_prefetch")]

    def as_dict(self) -> dict:
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["variant"] = VARIANT_NAMES.get(d["variant"], d["variant"])
        return d


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"RMSNorm CUDA library not built ({path} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
            L.rmsnorm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, f32, f32, i32, vp]
            L.rmsnorm_fwd.restype = i32
            L.rmsnorm_fwd_ex.argtypes = [vp, vp, vp, vp, i64, i64, f32, f32, i32,
                                         ctypes.POINTER(Options), vp]
            L.rmsnorm_fwd_ex.restype = i32
            L.rmsnorm_fwd_strided.argtypes = [vp, i64, vp, vp, i64, vp, i64, i64, f32, f32, i32,
                                              ctypes.POINTER(Options), vp]
            L.rmsnorm_fwd_strided.restype = i32
            L.rmsnorm_fwd_host.argtypes = [vp, vp, vp, vp, i64, i64, f32, f32, i32, i64, vp, i64,
                                           ctypes.POINTER(Options), vp]
            L.rmsnorm_fwd_host.restype = i32
            L.rmsnorm_fwd_host_workspace_size.argtypes = [i64, i64, i32, i64,
                                                          ctypes.POINTER(ctypes.c_int64)]
            L.rmsnorm_fwd_host_workspace_size.restype = i32
            L.rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp, i64,
                                      ctypes.POINTER(Options), vp]
            L.rmsnorm_bwd.restype = i32
            L.rmsnorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f32, i32,
                                              ctypes.POINTER(Options), vp]
            L.rmsnorm_bwd_noalloc.restype = i32
            L.rmsnorm_bwd_workspace_size.argtypes = [i64, i64, i32, ctypes.POINTER(Options),
                                                     ctypes.POINTER(ctypes.c_int64)]
            L.rmsnorm_bwd_workspace_size.restype = i32
            L.rmsnorm_plan_info.argtypes = [i64, i64, i32, vp, vp, vp, ctypes.POINTER(Options),
                                            ctypes.POINTER(Plan)]
            L.rmsnorm_plan_info.restype = i32
            L.rmsnorm_bwd_plan_info.argtypes = [i64, i64, i32, ctypes.POINTER(Options),
                                                ctypes.POINTER(Plan)]
            L.rmsnorm_bwd_plan_info.restype = i32
            L.rmsnorm_check_device_status.argtypes = [vp]
            L.rmsnorm_check_device_status.restype = i32
            L.rmsnorm_strerror.argtypes = [i32]
            L.rmsnorm_strerror.restype = ctypes.c_char_p
            L.rmsnorm_last_error.argtypes = []
            L.rmsnorm_last_error.restype = ctypes.c_char_p
            L.rmsnorm_version.argtypes = []
            L.rmsnorm_version.restype = i32
            _lib = L
    return _lib


def _check(rc: int) -> int:
    if rc != 0:
        raise RMSNormError(rc, lib().rmsnorm_last_error().decode())
    return rc


FLAG_NO_PDL = 1
FLAG_BLOCKED_ROWS = 2
FLAG_EARLY_LOADS = 4
FLAG_HOST_DIRECT = 8
FLAG_EARLY_WEIGHTS = 16
FLAG_BULK_STORE = 32


def make_options(variant: str | int = "auto", max_ctas: int = 0, lanes_per_row: int = 0,
                 stages: int = 0, rows_per_stage: int = 0, wait_limit_ns: int = 0,
                 pdl: bool = True, blocked: bool = False, early_loads: bool = False,
                 cluster_size: int = 0, host_direct: bool = False,
                 early_weights: bool = False, bulk_store: bool = False,
                 l2_prefetch: int = 0, prewait_prefetch: int = 0) -> Options:
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    flags = ((0 if pdl else FLAG_NO_PDL) | (FLAG_BLOCKED_ROWS if blocked else 0)
             | (FLAG_EARLY_LOADS if early_loads else 0) | (FLAG_HOST_DIRECT if host_direct else 0)
             | (FLAG_EARLY_WEIGHTS if early_weights else 0) | (FLAG_BULK_STORE if bulk_store else 0))
    return Options(ctypes.sizeof(Options), v, max_ctas, lanes_per_row, stages, rows_per_stage,
                   flags, cluster_size, wait_limit_ns, l2_prefetch, prewait_prefetch)


# ---- raw C ABI (integer device addresses) --------------------------------

def rmsnorm_fwd(x: int, w: int, y: int, rstd: int, M: int, N: int, eps: float, offset: float,
                dtype: int, stream: int) -> int:
    return lib().rmsnorm_fwd(x, w, y, rstd, M, N, eps, offset, dtype, stream)


def rmsnorm_fwd_ex(x: int, w: int, y: int, rstd: int, M: int, N: int, eps: float, offset: float,
                   dtype: int, opts: Options | None, stream: int) -> int:
    return lib().rmsnorm_fwd_ex(x, w, y, rstd, M, N, eps, offset, dtype,
                                ctypes.byref(opts) if opts is not None else None, stream)


def rmsnorm_fwd_strided(x: int, ldx: int, w: int, y: int, ldy: int, rstd: int, M: int, N: int,
                        eps: float, offset: float, dtype: int, opts: Options | None,
                        stream: int) -> int:
    return lib().rmsnorm_fwd_strided(x, ldx, w, y, ldy, rstd, M, N, eps, offset, dtype,
                                     ctypes.byref(opts) if opts is not None else None, stream)


def rmsnorm_fwd_host(x_host: int, w: int, y_host: int, rstd_host: int, M: int, N: int,
                     eps: float, offset: float, dtype: int, chunk_rows: int, workspace: int,
                     workspace_bytes: int, opts: Options | None, stream: int) -> int:
    """The forward over host-resident x/y/rstd (w and the workspace on the device)."""
    return lib().rmsnorm_fwd_host(x_host, w, y_host, rstd_host, M, N, eps, offset, dtype,
                                  chunk_rows, workspace, workspace_bytes,
                                  ctypes.byref(opts) if opts is not None else None, stream)


def rmsnorm_fwd_host_workspace_size(M: int, N: int, dtype: int, chunk_rows: int = 0) -> int:
    out = ctypes.c_int64(0)
    _check(lib().rmsnorm_fwd_host_workspace_size(M, N, dtype, chunk_rows, ctypes.byref(out)))
    return out.value


def rmsnorm_bwd(x: int, w: int, rstd: int, dy: int, dx: int, dw: int, M: int, N: int,
                offset: float, dtype: int, workspace: int, workspace_bytes: int,
                opts: Options | None, stream: int) -> int:
    return lib().rmsnorm_bwd(x, w, rstd, dy, dx, dw, M, N, offset, dtype, workspace,
                             workspace_bytes, ctypes.byref(opts) if opts is not None else None,
                             stream)


def rmsnorm_bwd_noalloc(x: int, w: int, rstd: int, dy: int, dx: int, dw: int, M: int, N: int,
                        offset: float, dtype: int, opts: Options | None, stream: int) -> int:
    """rmsnorm_bwd with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory at the call)."""
    return lib().rmsnorm_bwd_noalloc(x, w, rstd, dy, dx, dw, M, N, offset, dtype,
                                     ctypes.byref(opts) if opts is not None else None, stream)


def rmsnorm_bwd_workspace_size(M: int, N: int, dtype: int, opts: Options | None = None) -> int:
    out = ctypes.c_int64(0)
    _check(lib().rmsnorm_bwd_workspace_size(M, N, dtype,
                                            ctypes.byref(opts) if opts is not None else None,
                                            ctypes.byref(out)))
    return out.value


def rmsnorm_plan_info(M: int, N: int, dtype: int, x: int = 0, w: int = 0, y: int = 0,
                      opts: Options | None = None) -> dict:
    out = Plan()
    _check(lib().rmsnorm_plan_info(M, N, dtype, x, w, y,
                                   ctypes.byref(opts) if opts is not None else None,
                                   ctypes.byref(out)))
    return out.as_dict()


def rmsnorm_bwd_plan_info(M: int, N: int, dtype: int, opts: Options | None = None) -> dict:
    """The backward row kernel's launch for aligned buffers (no launch)."""
    out = Plan()
    _check(lib().rmsnorm_bwd_plan_info(M, N, dtype, ctypes.byref(opts) if opts is not None else None,
                                       ctypes.byref(out)))
    return out.as_dict()


def rmsnorm_check_device_status(stream: int = 0) -> int:
    return lib().rmsnorm_check_device_status(stream)


def rmsnorm_strerror(status: int) -> str:
    return lib().rmsnorm_strerror(status).decode()


def rmsnorm_last_error() -> str:
    return lib().rmsnorm_last_error().decode()


def rmsnorm_version() -> int:
    return lib().rmsnorm_version()


# ---- torch convenience ---------------------------------------------------

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"RMSNorm takes bf16, fp16 or fp32 activations, got {t.dtype}")


def fwd(x, w, eps: float = 1e-6, offset: float = 0.0, y=None, rstd=None, stream=None,
        **options):
    """y, rstd = fwd(x, w): RMSNorm forward of a contiguous CUDA tensor x[..., N].

    ``y`` and ``rstd`` may be passed to write in place (y may be x itself);
    ``rstd=False`` skips storing rstd (inference). 2-D ``x``/``y`` views with unit
    column stride (rows of wider tensors) go through ``rmsnorm_fwd_strided``.
    Keyword ``options`` go to :func:`make_options` (variant, max_ctas, ...).
    Runs on ``stream`` (a torch.cuda.Stream) or the current stream.
    """
    import torch
    if not (x.is_cuda and w.is_cuda):
        raise ValueError("x and w must be CUDA tensors")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    N = x.shape[-1]
    if w.dtype != x.dtype or w.numel() != N:
        raise ValueError("w must have x's dtype and N elements")
    if x.is_contiguous():
        M, ldx = (x.numel() // N if N else 0), N
    elif x.dim() == 2 and x.stride(1) == 1:
        M, ldx = x.shape[0], x.stride(0)  # rows of a wider tensor
    else:
        raise ValueError("x must be contiguous, or 2-D with unit column stride")
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    ldy = y.stride(0) if (y.dim() == 2 and not y.is_contiguous()) else N
    if y.shape != x.shape or (ldy == N and not y.is_contiguous()):
        raise ValueError("y must have x's shape, contiguous or 2-D with unit column stride")
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    r_ptr = 0 if rstd is False else rstd.data_ptr()
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    opts = make_options(**options) if options else None
    with torch.cuda.device(x.device):
        _check(rmsnorm_fwd_strided(x.data_ptr(), ldx, w.data_ptr(), y.data_ptr(), ldy, r_ptr, M,
                                   N, eps, offset, _dtype_code(x), opts, s.cuda_stream))
    return y, (None if rstd is False else rstd)


def fwd_host(x, w, eps: float = 1e-6, offset: float = 0.0, y=None, rstd=None,
             chunk_rows: int = 0, workspace=None, stream=None, **options):
    """y, rstd = fwd_host(x, w): the forward of a contiguous CPU tensor x[..., N]
    (pinned for overlapped copies) with w on the GPU, through rmsnorm_fwd_host.

    ``y`` and ``rstd`` are CPU tensors (allocated pinned when not given; y may be
    x itself); ``rstd=False`` skips rstd. The device ``workspace`` (a CUDA tensor)
    is allocated here with torch when not given (none with ``host_direct=True``:
    the kernel then reads and writes the pinned host buffers itself). The call
    is asynchronous on
    ``stream`` (or the current stream of w's device): synchronise before reading.
    """
    import torch
    if x.is_cuda or not w.is_cuda:
        raise ValueError("x must be a CPU tensor and w a CUDA tensor")
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous")
    N = x.shape[-1]
    if w.dtype != x.dtype or w.numel() != N:
        raise ValueError("w must have x's dtype and N elements")
    M = x.numel() // N if N else 0
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    if y.shape != x.shape or y.dtype != x.dtype or y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CPU tensor like x")
    if rstd is None:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32).pin_memory()
    r_ptr = 0 if rstd is False else rstd.data_ptr()
    code = _dtype_code(x)
    opts = make_options(**options) if options else None
    with torch.cuda.device(w.device):
        need = rmsnorm_fwd_host_workspace_size(M, N, code, chunk_rows)
        if workspace is None and not options.get("host_direct"):
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=w.device)
        s = stream if stream is not None else torch.cuda.current_stream(w.device)
        ws_ptr = 0 if workspace is None else workspace.data_ptr()
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(rmsnorm_fwd_host(x.data_ptr(), w.data_ptr(), y.data_ptr(), r_ptr, M, N, eps,
                                offset, code, chunk_rows, ws_ptr, ws_bytes, opts, s.cuda_stream))
    return y, (None if rstd is False else rstd)


def bwd(x, w, rstd, dy, offset: float = 0.0, dx=None, stream=None, **options):
    """dx, dw = bwd(x, w, rstd, dy): backward of ``fwd`` for contiguous CUDA tensors.

    The fp32 workspace for the dw partials is allocated here with torch (the C
    library never allocates); dw comes back in fp32.
    """
    import torch
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    if dx is None:
        dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=x.device)
    opts = make_options(**options) if options else None
    with torch.cuda.device(x.device):
        nbytes = rmsnorm_bwd_workspace_size(M, N, _dtype_code(x), opts)
        ws = torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32, device=x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        _check(rmsnorm_bwd(x.data_ptr(), w.data_ptr(), rstd.data_ptr(), dy.data_ptr(),
                           dx.data_ptr(), dw.data_ptr(), M, N, offset, _dtype_code(x),
                           ws.data_ptr(), ws.numel() * 4, opts, s.cuda_stream))
        # The workspace was allocated on the current stream; keep it from being
        # reused before the work on `s` is done.
        ws.record_stream(s)
    return dx, dw
