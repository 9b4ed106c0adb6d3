"""Padding study of the planner on synthetic MoE layer groups.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §6.4 (Figure 11):
with row granularity 1x or 16x the planned buffers carry under 3% padding at
every FSDP size, while at 128 rows (128x128 tiling) a model whose experts are
fused into one parameter tensor per projection shows step-like spikes of up to
18%, and a model with one tensor per expert stays low (its tensors leave the
planner more places to cut).  §5 (Planning algorithm): the default tensor order
was compared with block-size and shape orders.

The pages do not list the models' shapes, so the groups here are synthetic
transformer-MoE layers with the two expert layouts:
  fused       wq, wk, wv, wo, router, experts.gate_up [E*2f, d],
              experts.down [E*d, f], two norm vectors;
  per-expert  the same attention and router, then gate [f, d], up [f, d] and
              down [d, f] for every expert.
Every matrix is sharded at `gran` rows; vectors at single elements.  Padding
is (m*S - E) / E, the buffer inflation over the group's elements.

Run ``python -m fsdp_infra_gb300.padding_study`` for the markdown tables.
"""
from __future__ import annotations

import argparse
import time
from typing import Dict, List, Sequence, Tuple

from . import dbuf as _c

Spec = Tuple[int, int, int]   # rows, cols, gran_rows

FSDP_SIZES = (8, 16, 32, 64, 128, 256, 512, 1024)
GRANULARITIES = (1, 16, 128)


def moe_layer(style: str, experts: int, d: int, f: int, d_kv: int, gran: int) -> List[Spec]:
    """One synthetic MoE transformer layer as planner specs (rows, cols, gran)."""
    attn = [(d, d, gran), (d_kv, d, gran), (d_kv, d, gran), (d, d, gran), (experts, d, gran)]
    norms = [(d, 1, 1), (d, 1, 1)]
    if style == "fused":
        moe = [(experts * 2 * f, d, gran), (experts * d, f, gran)]
    elif style == "per_expert":
        moe = []
        for _ in range(experts):
            moe += [(f, d, gran), (f, d, gran), (d, f, gran)]
    else:
        raise ValueError(style)
    return attn + moe + norms


# Two synthetic models: experts fused into single tensors (fewer, larger
# experts), and many small experts kept as separate tensors.
MODELS: Dict[str, dict] = {
    "fused": dict(style="fused", experts=128, d=2880, f=2880, d_kv=512),
    "per_expert": dict(style="per_expert", experts=256, d=7168, f=2048, d_kv=1536),
}


def plan_padding(specs: Sequence[Spec], m: int, align: int = 16) -> Tuple[int, float, float]:
    """(S, padding %, planner ms) of one group."""
    t0 = time.perf_counter()
    p = _c.dbuf_plan(list(specs), m, None, align)
    ms = (time.perf_counter() - t0) * 1e3
    try:
        q = _c.dbuf_plan_query(p, len(specs), m)
    finally:
        _c.dbuf_plan_free(p)
    e = sum(r * c for r, c, _ in specs)
    return q["S"], 100.0 * (m * q["S"] - e) / e, ms


def sweep(models=MODELS, sizes=FSDP_SIZES, grans=GRANULARITIES) -> List[dict]:
    rows = []
    for name, cfg in models.items():
        for g in grans:
            specs = moe_layer(gran=g, **cfg)
            for m in sizes:
                S, pad, ms = plan_padding(specs, m)
                rows.append({"model": name, "gran": g, "m": m, "S": S, "padding_pct": pad,
                             "planner_ms": ms, "tensors": len(specs)})
    return rows


def order_study(groups: Dict[str, Tuple[Sequence[Spec], int]]) -> List[dict]:
    """S under the three orders for each (specs, m)."""
    out = []
    for name, (specs, m) in groups.items():
        row = {"group": name, "m": m}
        for kind in ("default", "block", "shape"):
            perm = _c.dbuf_order(list(specs), kind)
            S, pad, _ = plan_padding([specs[i] for i in perm], m)
            row[kind] = (S, pad)
        out.append(row)
    return out


def _markdown(rows: List[dict], sizes=FSDP_SIZES) -> str:
    lines = ["| model | gran rows | " + " | ".join(f"m={m}" for m in sizes) + " | max |",
             "|---|---|" + "---|" * (len(sizes) + 1)]
    keys = sorted({(r["model"], r["gran"]) for r in rows}, key=lambda k: (k[0], k[1]))
    for model, g in keys:
        sel = {r["m"]: r["padding_pct"] for r in rows if r["model"] == model and r["gran"] == g}
        vals = [sel[m] for m in sizes]
        lines.append(f"| {model} | {g} | " + " | ".join(f"{v:.2f}%" for v in vals) +
                     f" | {max(vals):.2f}% |")
    return "\n".join(lines)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--orders", action="store_true", help="also compare the three orders")
    args = ap.parse_args(argv)
    t0 = time.perf_counter()
    rows = sweep()
    print("padding (m*S - E) / E of one synthetic MoE layer group, planner default order\n")
    print(_markdown(rows))
    worst = max(r["planner_ms"] for r in rows)
    print(f"\nslowest plan: {worst:.1f} ms; sweep {time.perf_counter() - t0:.1f} s")
    if args.orders:
        groups = {}
        for name, cfg in MODELS.items():
            for g in GRANULARITIES:
                for m in (64, 1024):
                    groups[f"{name} gran={g}"] = (moe_layer(gran=g, **cfg), m)
                    groups[f"{name} gran={g} m={m}"] = groups.pop(f"{name} gran={g}")
        print("\n| group | default S (pad) | block-size S (pad) | shape S (pad) |\n|---|---|---|---|")
        for r in order_study(groups):
            cells = [f"{r[k][0]} ({r[k][1]:.2f}%)" for k in ("default", "block", "shape")]
            print(f"| {r['group']} | " + " | ".join(cells) + " |")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
