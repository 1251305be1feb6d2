"""fp64 CPU oracle for the RMSNorm forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does, and this
package imports nothing from it: the two share no code.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, fp64, compiled with gcc
without fast-math or FMA contraction). This module compiles it on demand and
marshals numpy arrays through ctypes. Definitions and sources are in the C
file's header: the TileGym issue #169 kernel listing ("Why cutile's rmsnorm
required full register") and the skillmd "RMSNorm Kernel Optimization" page
(Overview, Verification).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_LIB = os.path.join(_HERE, "librmsnorm_oracle.so")
_DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}
# Bit-pattern container per dtype: 16-bit formats in uint16, fp32 in uint32.
_BITS = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.uint32}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/librmsnorm_oracle.so`` (gcc, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp = ctypes.c_void_p
            f64p = ctypes.POINTER(ctypes.c_double)
            L.oracle_rmsnorm_fwd.argtypes = [vp, vp, vp, f64p, f64p, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                             ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
            L.oracle_rmsnorm_fwd.restype = ctypes.c_int
            L.oracle_rmsnorm_bwd.argtypes = [vp, vp, vp, f64p, vp, f64p, f64p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                             ctypes.c_float, ctypes.c_int]
            L.oracle_rmsnorm_bwd.restype = ctypes.c_int
            L.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_int64, vp, f64p]
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_encode.argtypes = [ctypes.c_int, ctypes.c_int64, f64p, vp]
            L.oracle_encode.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.POINTER(ctype)()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _vp(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def bits_dtype(dtype: str):
    """numpy container of the bit patterns of ``dtype`` (uint16 or uint32)."""
    return _BITS[dtype]


def decode(dtype: str, bits: np.ndarray) -> np.ndarray:
    """bf16/fp16 (uint16) or fp32 (uint32) bit patterns -> exact float64 values."""
    bits = np.ascontiguousarray(bits, dtype=_BITS[dtype])
    out = np.empty(bits.shape, dtype=np.float64)
    rc = lib().oracle_decode(_DTYPES[dtype], bits.size, _vp(bits), _ptr(out, ctypes.c_double))
    assert rc == 0
    return out


def encode(dtype: str, values: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16/fp16/fp32 bit pattern, ties to even."""
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=_BITS[dtype])
    rc = lib().oracle_encode(_DTYPES[dtype], values.size, _ptr(values, ctypes.c_double), _vp(out))
    assert rc == 0
    return out


def rmsnorm_fwd(x_bits: np.ndarray, w_bits: np.ndarray, eps: float, offset: float, dtype: str,
                rows: tuple[int, int] | None = None, want_y64: bool = False):
    """RMSNorm forward over rows ``[r0, r1)`` of ``x_bits`` ([M, N] bit patterns).

    Returns ``(y_bits, rstd_f64)`` for those rows, plus the unrounded fp64 y
    when ``want_y64``. ``eps`` and ``offset`` are taken as fp32, as the CUDA
    entry point takes them.
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=_BITS[dtype])
    w_bits = np.ascontiguousarray(w_bits, dtype=_BITS[dtype])
    M, N = x_bits.shape
    assert w_bits.shape == (N,)
    r0, r1 = (0, M) if rows is None else rows
    y = np.zeros((M, N), dtype=_BITS[dtype]) if rows is None else None
    rstd = np.zeros(M, dtype=np.float64)
    y64 = np.zeros((M, N), dtype=np.float64) if want_y64 else None
    if rows is not None:
        # Work on the slice only, so a row range costs only its own rows.
        xs = np.ascontiguousarray(x_bits[r0:r1])
        return rmsnorm_fwd(xs, w_bits, eps, offset, dtype, None, want_y64)
    rc = lib().oracle_rmsnorm_fwd(_vp(x_bits), _vp(w_bits), _vp(y), _ptr(rstd, ctypes.c_double),
                                  _ptr(y64, ctypes.c_double), M, N, eps, offset, _DTYPES[dtype],
                                  r0, r1)
    assert rc == 0
    return (y, rstd, y64) if want_y64 else (y, rstd)


def rmsnorm_fwd_into(x_bits: np.ndarray, w_bits: np.ndarray, y_out: np.ndarray,
                     rstd_out: np.ndarray, eps: float, offset: float, dtype: str,
                     row0: int, row1: int) -> None:
    """Rows ``[row0, row1)`` written into caller-owned arrays (used for threaded runs:
    ctypes releases the GIL for the duration of the C call)."""
    M, N = x_bits.shape
    for a in (x_bits, w_bits, y_out):
        assert a.dtype == _BITS[dtype]
    rc = lib().oracle_rmsnorm_fwd(_vp(x_bits), _vp(w_bits), _vp(y_out),
                                  _ptr(rstd_out, ctypes.c_double), None, M, N, eps, offset,
                                  _DTYPES[dtype], row0, row1)
    assert rc == 0


def rmsnorm_bwd(x_bits: np.ndarray, w_bits: np.ndarray, dy_bits: np.ndarray, offset: float,
                dtype: str, rstd: np.ndarray | None = None, eps: float = 0.0):
    """Backward of the forward above (derived by the chain rule; see the C file).

    ``rstd`` (per row, any float array) is the saved rstd the backward consumes;
    None recomputes it in fp64 from x and ``eps``. Returns ``(dx_bits, dx_f64,
    dw_f64)``.
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=_BITS[dtype])
    dy_bits = np.ascontiguousarray(dy_bits, dtype=_BITS[dtype])
    w_bits = np.ascontiguousarray(w_bits, dtype=_BITS[dtype])
    M, N = x_bits.shape
    assert dy_bits.shape == (M, N) and w_bits.shape == (N,)
    r = None if rstd is None else np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.zeros((M, N), dtype=_BITS[dtype])
    dx64 = np.zeros((M, N), dtype=np.float64)
    dw = np.zeros(N, dtype=np.float64)
    rc = lib().oracle_rmsnorm_bwd(_vp(x_bits), _vp(w_bits), _vp(dy_bits), _ptr(r, ctypes.c_double),
                                  _vp(dx), _ptr(dx64, ctypes.c_double), _ptr(dw, ctypes.c_double),
                                  M, N, eps, offset, _DTYPES[dtype])
    assert rc == 0
    return dx, dx64, dw
