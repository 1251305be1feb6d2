"""Seeded synthetic inputs for the RMSNorm forward.

This module draws random numbers and nothing else: it holds none of the
normalisation's arithmetic, so both the CUDA path's tests/benchmark and the
fp64 oracle take their inputs from here.

Recipe (every workload): one ``torch.Generator('cpu')`` seeded with the
workload's seed; x is drawn first, in blocks of rows (block = max(1, 2**22 // N)
rows, each block drawn in full before the next), then w. Values are drawn in
fp32 and rounded to the activation dtype by torch's ``.to()`` (round to nearest
even). Arrays come back as raw bit patterns: uint16 for bf16/fp16, uint32 for
fp32 (drawn in fp32, so no rounding at all).

The five named workloads reproduce the shapes and distributions the method is
benchmarked on: the 16384x512 bf16 shape reported for the persistent cuTile
kernel (TileGym issue #169), plus a small case, a non-power-of-two hidden size
with Gemma-style weights (offset 1), a large hidden size with heavy-tailed
activations, and a large fp16 case whose sum of squares exceeds the fp16 range.
``N(mu, v)`` below means variance ``v``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = ("bf16", "fp16", "fp32")
_TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
_INT = {"bf16": (torch.int16, np.uint16), "fp16": (torch.int16, np.uint16),
        "fp32": (torch.int32, np.uint32)}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    dtype: str = "bf16"
    x_std: float = 1.0            # x ~ N(0, x_std^2)
    outlier_p: float = 0.0        # heavy tail: with probability p, x ~ N(0, outlier_std^2)
    outlier_std: float = 100.0
    w_kind: str = "uniform"       # "uniform": U(w_a, w_b); "normal": N(w_a, w_b)
    w_a: float = 0.5
    w_b: float = 1.5
    eps: float = 1e-6
    offset: float = 0.0
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes one forward must move: x read, y written, w read, rstd written."""
        e = ELEM_BYTES[self.dtype]
        return e * self.M * self.N + e * self.M * self.N + e * self.N + 4 * self.M


WORKLOADS = {
    w.name: w
    for w in [
        Workload("rmsnorm_2048x512_bf16", 2048, 512, note="small case"),
        Workload("rmsnorm_16384x512_bf16", 16384, 512,
                 note="the shape of the persistent cuTile kernel report"),
        Workload("rmsnorm_32768x1000_bf16_gemma", 32768, 1000, w_kind="normal", w_a=0.0,
                 w_b=0.1, offset=1.0, note="non-power-of-two N, masked tail, Gemma offset"),
        Workload("rmsnorm_16384x8192_bf16_heavytail", 16384, 8192, outlier_p=0.01,
                 outlier_std=100.0, eps=1e-5, note="99% N(0,1) + 1% N(0,100^2)"),
        Workload("rmsnorm_131072x4096_fp16", 131072, 4096, dtype="fp16", x_std=64.0,
                 note="sum of squares far beyond the fp16 range"),
    ]
}
BENCH_WORKLOAD = "rmsnorm_16384x512_bf16"

# fp32 activations (x, w, y in fp32) at the benchmark shapes: not among the
# named workloads above, which are the method's own; measured and tested as a
# boundary variant of the same forward. Also one smaller size of a named
# workload for profiler captures.
EXTRA_WORKLOADS = {
    w.name: w
    for w in [
        Workload("rmsnorm_16384x512_fp32", 16384, 512, dtype="fp32"),
        Workload("rmsnorm_32768x1000_fp32_gemma", 32768, 1000, dtype="fp32", w_kind="normal",
                 w_a=0.0, w_b=0.1, offset=1.0),
        Workload("rmsnorm_16384x8192_fp32_heavytail", 16384, 8192, dtype="fp32", outlier_p=0.01,
                 outlier_std=100.0, eps=1e-5),
        Workload("rmsnorm_65536x4096_fp32", 65536, 4096, dtype="fp32", x_std=64.0),
        # The 131072x4096 fp16 workload's kernel and plan at an eighth of its
        # rows (x 128 MB, still above L2), for profiler captures of one launch.
        Workload("rmsnorm_16384x4096_fp16", 16384, 4096, dtype="fp16", x_std=64.0),
    ]
}


def get(name: str) -> Workload:
    """A named workload, or one of the extra ones (fp32, profiling size)."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    return EXTRA_WORKLOADS[name]


def _bits(t: torch.Tensor, dtype: str) -> np.ndarray:
    ti, ni = _INT[dtype]
    return t.to(_TORCH[dtype]).view(ti).numpy().view(ni)


def generate(wl: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Return ``(x_bits [M, N], w_bits [N])`` for the workload (uint16, or uint32 for fp32)."""
    M = wl.M
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed)
    x = np.empty((M, wl.N), dtype=_INT[wl.dtype][1])
    block = max(1, (1 << 22) // wl.N)
    for r0 in range(0, M, block):
        r1 = min(M, r0 + block)
        t = torch.randn((r1 - r0, wl.N), generator=g, dtype=torch.float32) * wl.x_std
        if wl.outlier_p > 0.0:
            mask = torch.rand((r1 - r0, wl.N), generator=g) < wl.outlier_p
            out = torch.randn((r1 - r0, wl.N), generator=g, dtype=torch.float32) * wl.outlier_std
            t = torch.where(mask, out, t)
        x[r0:r1] = _bits(t, wl.dtype)
    if wl.w_kind == "uniform":
        w = wl.w_a + (wl.w_b - wl.w_a) * torch.rand(wl.N, generator=g, dtype=torch.float32)
    elif wl.w_kind == "normal":
        w = wl.w_a + (wl.w_b ** 0.5) * torch.randn(wl.N, generator=g, dtype=torch.float32)
    else:
        raise ValueError(wl.w_kind)
    return x, _bits(w, wl.dtype)


def custom(M: int, N: int, dtype: str = "bf16", seed: int = 0, **kw) -> Workload:
    """An ad-hoc workload (parity sweeps over small and ragged shapes)."""
    return Workload(f"custom_{M}x{N}_{dtype}_s{seed}", M, N, dtype=dtype, seed=seed, **kw)


def to_torch(bits: np.ndarray, dtype: str) -> torch.Tensor:
    """Bit patterns -> a CPU torch tensor of the activation dtype (no copy of values)."""
    signed = np.int32 if dtype == "fp32" else np.int16
    return torch.from_numpy(np.ascontiguousarray(bits).view(signed)).view(_TORCH[dtype])


def from_torch(t: torch.Tensor) -> np.ndarray:
    """A bf16/fp16/fp32 torch tensor (any device) -> its bit patterns on the host."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)
