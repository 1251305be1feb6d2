"""Parity report (run on a GPU): for each workload, the CUDA forward in the
automatic launch (both launch modes the benchmark times) against the fp64
oracle: max ulp and a histogram of ulp distances of y, and the max relative
error of rstd. Prints a markdown table.

    python tests/parity_report.py [--rows-cap N]

Rows: all of them for workloads of up to 2^25 elements, else `--rows-cap`
sampled rows (first, middle, last and random ones). fp32 workloads report the
ulp distance from the correctly rounded fp64 value (the kernels' fp32 product
is within a few ulps; the tests check the derived bound).
"""
from __future__ import annotations

import argparse
import collections
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from memory_bound_normalization_fwd_gb300 import binding as B  # noqa: E402
from memory_bound_normalization_fwd_gb300 import workloads as W  # noqa: E402
from parity_util import DT, DeviceCase, ordinal, ordinal32, sample_rows  # noqa: E402


def report(wl, early: bool, rows_cap: int):
    x, w = W.generate(wl)
    rows = None if wl.M * wl.N <= (1 << 25) else sample_rows(wl.M, rows_cap, seed=3)
    case = DeviceCase(x, w, wl.dtype)
    for _ in range(2 if early else 1):
        assert case.run(wl.eps, wl.offset, early_loads=early) == 0, B.rmsnorm_last_error()
    y, r = case.results()
    case.check_guards()
    xs = x if rows is None else np.ascontiguousarray(x[rows])
    yo, ro = oracle.rmsnorm_fwd(xs, w, wl.eps, wl.offset, wl.dtype)
    if rows is not None:
        y, r = y[rows], r[rows]
    if wl.dtype == "fp32":
        d = np.abs(ordinal32(y) - ordinal32(yo))
    else:
        d = np.abs(ordinal(y) - ordinal(yo))
    hist = collections.Counter(d.ravel().tolist())
    rel = np.abs(r.astype(np.float64) - ro) / np.abs(ro)
    plan = B.rmsnorm_plan_info(wl.M, wl.N, DT[wl.dtype], case.x.data_ptr(), case.w.data_ptr(),
                               case.y.data_ptr(), B.make_options(early_loads=early))
    return {"rows": wl.M if rows is None else len(rows), "max_ulp": int(d.max()),
            "hist": dict(sorted(hist.items())), "max_rstd_rel": float(rel.max()),
            "variant": plan["variant"]}


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--rows-cap", type=int, default=2048)
    args = p.parse_args(argv)
    wls = list(W.WORKLOADS.values()) + list(W.EXTRA_WORKLOADS.values())
    print("| workload | launch | kernel | rows checked | max ulp | ulp histogram (distance: count) | max rstd rel err |")
    print("|---|---|---|---|---|---|---|")
    for wl in wls:
        for early in (False, True):
            r = report(wl, early, args.rows_cap)
            hist = ", ".join(f"{k}: {v}" for k, v in r["hist"].items())
            print(f"| {wl.name} | {'early loads' if early else 'strict'} | {r['variant']} | "
                  f"{r['rows']} | {r['max_ulp']} | {hist} | {r['max_rstd_rel']:.2e} |", flush=True)
            torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
