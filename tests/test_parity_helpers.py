"""Host checks of the parity helpers the full-size GPU tests rely on: the
threaded oracle gives the single-call oracle's bits, and the block-wise
comparison finds a difference in any block and counts ulp distances exactly."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from memory_bound_normalization_fwd_gb300 import workloads as W
from parity_util import compare_blocked, oracle_threaded


@pytest.mark.parametrize("M,N,dtype,threads", [(1, 8, "bf16", 4), (37, 1000, "bf16", 5),
                                               (130, 520, "fp16", 3), (64, 24, "fp32", 64)])
def test_threaded_oracle_equals_one_call(M, N, dtype, threads):
    wl = W.custom(M, N, dtype, seed=M + N, offset=1.0)
    x, w = W.generate(wl)
    y1, r1 = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, dtype)
    y2, r2 = oracle_threaded(x, w, wl.eps, wl.offset, dtype, threads=threads)
    assert np.array_equal(y1, y2) and np.array_equal(r1, r2)


def test_compare_blocked_counts_and_catches_every_block():
    wl = W.custom(50, 16, "bf16", seed=3)
    x, w = W.generate(wl)
    y, r = oracle.rmsnorm_fwd(x, w, wl.eps, wl.offset, "bf16")
    g = y.copy()
    g[7, 3] += 1      # one ulp up (positive value or not, a neighbour in value order)
    u, e, hist = compare_blocked(g, r.astype(np.float32), y, r, "bf16", block_elems=64)
    assert u == 1 and e <= 1e-7
    assert hist == {0: 50 * 16 - 1, 1: 1}
    for row in (0, 23, 49):  # a 2-ulp slip in the first, a middle or the last block fails
        bad = y.copy()
        bad[row, 5] += 2
        with pytest.raises(AssertionError):
            compare_blocked(bad, r, y, r, "bf16", block_elems=64)
    rb = r.copy()
    rb[49] *= 1 + 2e-5
    with pytest.raises(AssertionError):
        compare_blocked(y, rb, y, r, "bf16", block_elems=64)
