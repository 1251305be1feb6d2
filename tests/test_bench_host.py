"""Host logic of bench.py that needs no GPU: which committed traffic figure
the benchmark line may quote."""
from __future__ import annotations

import json

import bench

PLAN = {"variant": "tma", "threads": 256, "grid": 456, "lanes_per_row": 16, "vecs_per_lane": 4,
        "rows_per_stage": 16, "stages": 2, "smem_bytes": 33024, "ctas_per_sm": 3,
        "sm_count": 152, "cluster_size": 0}


def _write(d, workload, h, plan, nbytes=123456):
    (d / f"traffic_{workload}.md").write_text(
        f"kernel_hash: `{h}`\ntraffic_bytes_per_launch: `{nbytes}`\nplan: `{json.dumps(plan)}`\n")


def test_traffic_needs_matching_kernel_sources_and_plan(tmp_path):
    d = str(tmp_path)
    _write(tmp_path, "w", bench.kernel_hash("tma"), PLAN)
    assert bench.load_traffic("w", PLAN, d) == 123456
    assert bench.load_traffic("w", dict(PLAN, grid=608), d) is None        # another launch
    assert bench.load_traffic("w", dict(PLAN, variant="warp"), d) is None  # another kernel
    assert bench.load_traffic("w", dict(PLAN, ctas_per_sm=4), d) == 123456  # not a launch field
    _write(tmp_path, "w", "0" * 16, PLAN)
    assert bench.load_traffic("w", PLAN, d) is None                        # sources changed
    assert bench.load_traffic("missing", PLAN, d) is None


def test_variant_hashes_cover_their_own_sources():
    assert len({bench.kernel_hash(v) for v in bench.VARIANT_SOURCES}) == len(bench.VARIANT_SOURCES)
    assert bench.kernel_hash("tma") != bench.kernel_hash()


def test_agree_allows_one_ulp_and_nothing_more():
    import numpy as np
    a = np.array([0x3F80, 0x8001, 0x0000, 0x7F7F], dtype=np.uint16)
    assert bench.agree(a, a.copy(), "bf16")
    assert bench.agree(a, np.array([0x3F81, 0x8001, 0x8000, 0x7F7F], dtype=np.uint16), "bf16")
    assert bench.agree(a, np.array([0x3F80, 0x0000, 0x0000, 0x7F7F], dtype=np.uint16), "bf16")
    assert not bench.agree(a, np.array([0x3F82, 0x8001, 0x0000, 0x7F7F], dtype=np.uint16), "bf16")
    f = np.array([1.0, -2.5], dtype=np.float32).view(np.uint32)
    assert bench.agree(f, f + 64, "fp32") and not bench.agree(f, f + 65, "fp32")
