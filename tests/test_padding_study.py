"""The padding study of the planner on synthetic MoE layers (host only).

Checks what the study reports: every plan it makes satisfies the layout
constraints; padding at 1x and 16x row granularity stays under 3% at every
FSDP size, as "veScale-FSDP" §6.4 reports; 128-row granularity is where
step-like padding appears; every plan takes under the pages' 0.3 s; the three
orders give valid plans and block-size order can beat the default one.
"""
from collections import namedtuple

from layout_check import check_layout

Spec = namedtuple("Spec", "rows cols gran_rows")


def _valid(dbuf_lib, specs, m):
    p = dbuf_lib.dbuf_plan(list(specs), m, None, 16)
    try:
        q = dbuf_lib.dbuf_plan_query(p, len(specs), m)
    finally:
        dbuf_lib.dbuf_plan_free(p)
    errs = check_layout([Spec(*s) for s in specs], q["offsets"], q["shard_bounds"], 16)
    assert not errs, errs[:3]
    return q["S"]


def test_sweep_plans_are_valid_and_fast(dbuf_lib):
    from fsdp_infra_gb300 import padding_study as ps
    rows = ps.sweep(sizes=(8, 64, 1024))
    assert len(rows) == 2 * 3 * 3
    for r in rows:
        assert r["padding_pct"] >= 0.0
        if r["planner_ms"] >= 300.0:
            # One wall-clock sample on a busy host can stall (page-in, another
            # process); the claim is about the planner, so take the best of three.
            specs = ps.moe_layer(gran=r["gran"], **ps.MODELS[r["model"]])
            r["planner_ms"] = min([r["planner_ms"]] +
                                  [ps.plan_padding(specs, r["m"])[2] for _ in range(2)])
        assert r["planner_ms"] < 300.0, r
        if r["gran"] in (1, 16):
            assert r["padding_pct"] < 3.0, r
    assert max(r["padding_pct"] for r in rows if r["gran"] == 128) > 3.0
    # spot-check the layouts themselves
    for name, cfg in ps.MODELS.items():
        specs = ps.moe_layer(gran=128, **cfg)
        S = _valid(dbuf_lib, specs, 1024)
        assert S == next(r["S"] for r in rows if r["model"] == name and r["gran"] == 128
                         and r["m"] == 1024)


def test_orders_give_valid_plans(dbuf_lib):
    from fsdp_infra_gb300 import padding_study as ps
    specs = ps.moe_layer(gran=128, **ps.MODELS["per_expert"])
    S = {}
    for kind in ("default", "block", "shape"):
        perm = dbuf_lib.dbuf_order(specs, kind)
        S[kind] = _valid(dbuf_lib, [specs[i] for i in perm], 1024)
    assert S["block"] < S["default"]
