"""Host logic of bench.py that needs no GPU: which committed traffic figure
the benchmark line may quote, the bit-agreement rule, and the reference arm
(the oracle timed on the host cores) with its JSON line."""
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


def test_traffic_file_with_one_entry_per_launch_plan(tmp_path):
    # Both launch modes of one workload in one summary: each plan finds its own figure.
    strict = dict(PLAN, variant="warp", grid=760, lanes_per_row=32, vecs_per_lane=2,
                  rows_per_stage=0, stages=1, smem_bytes=2048)
    (tmp_path / "traffic_w.md").write_text(
        f"## early\nkernel_hash: `{bench.kernel_hash('tma')}`\nplan: `{json.dumps(PLAN)}`\n"
        f"traffic_bytes_per_launch: `111`\n\n## strict\nkernel_hash: `{bench.kernel_hash('warp')}`\n"
        f"plan: `{json.dumps(strict)}`\ntraffic_bytes_per_launch: `222`\n")
    d = str(tmp_path)
    assert bench.load_traffic("w", PLAN, d) == 111
    assert bench.load_traffic("w", strict, d) == 222
    assert bench.load_traffic("w", dict(strict, grid=608), d) is None


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


def _reference_arm(env_extra):
    import os
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    root = os.path.dirname(os.path.abspath(bench.__file__))
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                           "--workload", "rmsnorm_2048x512_bf16", "--steps", "3", "--warmup", "3"],
                          capture_output=True, text=True, env=env, cwd=root, timeout=300)


def test_reference_arm_prints_one_contract_line_on_the_host():
    # The reference arm is the oracle on the host cores: no GPU, one JSON line
    # with the metric, unit and direction of the main arm, and the extra keys.
    p = _reference_arm({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] >= 3
    assert d["value"] > 0 and d["config"]["workload"] == "rmsnorm_2048x512_bf16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    p = _reference_arm({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
