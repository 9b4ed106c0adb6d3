"""Writes tests/golden/workload_plans.json from the oracle only.

Usage: python tests/golden/make_golden.py
The stored plan sizes are a regression guard for the five synthetic workloads;
they are computed by the oracle planner and by nothing else.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import WORKLOADS, workload  # noqa: E402


def main():
    out = {}
    for key in WORKLOADS:
        w = workload(key)
        groups = []
        for g in w.groups:
            p = oracle.plan_specs(g.tensors, w.m, w.local_units, w.align)
            groups.append({"group": g.name, "S": p.S, "total": p.total, "numel": g.numel,
                           "padding_pct": round(100.0 * (p.total - g.numel) / g.numel, 4)})
        out[key] = groups
    with open(os.path.join(HERE, "workload_plans.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
