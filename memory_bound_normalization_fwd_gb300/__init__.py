"""GB300 (sm_103a) RMSNorm forward: y = x * rsqrt(mean(x^2) + eps) * (offset + w),
with the per-row fp32 rstd kept for backward.

The computation runs in hand-written CUDA kernels behind the C ABI of
``include/rmsnorm.h`` (``librmsnorm_gb300.so``); this package is the ctypes
binding (:mod:`.binding`), the in-tree build step (:mod:`.build`) and the
seeded input generator (:mod:`.workloads`).
"""
from .binding import (  # noqa: F401
    BF16, FP16, EXPORTS, VARIANTS, Options, RMSNormError, bwd, fwd, lib, make_options,
    rmsnorm_bwd, rmsnorm_bwd_workspace_size,
    rmsnorm_check_device_status, rmsnorm_fwd, rmsnorm_fwd_ex, rmsnorm_fwd_strided, rmsnorm_last_error,
    rmsnorm_plan_info, rmsnorm_strerror, rmsnorm_version,
)
