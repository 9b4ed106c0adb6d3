"""The C++ planner in libdbuf equals the oracle byte for byte (S, offsets, shard
bounds, scale offsets, 8-bit optimizer state offsets) on the five workloads and on random groups, and plans
within the pages' runtime figure (under 0.3 s) -- host only, no GPU."""
import random
import time

import pytest

from workloads import WORKLOADS, workload
from workloads.configs import TensorSpec, random_tiny_group


def _cplan(d, specs, m, units=None, align=16):
    p = d.dbuf_plan(specs, m, units, align)
    try:
        q = d.dbuf_plan_query(p, len(specs), m)
        q["state_offsets"], q["n_state"] = d.dbuf_plan_state_offsets(p, len(specs))
        return q
    finally:
        d.dbuf_plan_free(p)


def _same(q, o, specs, oracle_lib):
    assert q["S"] == o.S
    assert q["total"] == o.total
    assert q["offsets"] == [int(x) for x in o.offsets]
    assert q["shard_bounds"] == [int(x) for x in o.bounds]
    soff, ns = oracle_lib.scale_offsets(specs)
    assert q["scale_offsets"] == [int(x) for x in soff] and q["n_scales"] == ns
    st, nst = oracle_lib.state_offsets(specs)
    assert q["state_offsets"] == [int(x) for x in st] and q["n_state"] == nst


@pytest.mark.parametrize("key", list(WORKLOADS))
def test_workloads_match_oracle(dbuf_lib, oracle_lib, oracle_plans, key):
    w = workload(key)
    for gi, g in enumerate(w.groups):
        t0 = time.perf_counter()
        q = _cplan(dbuf_lib, g.tensors, w.m, w.local_units, w.align)
        dt = time.perf_counter() - t0
        _same(q, oracle_plans(key, gi), g.tensors, oracle_lib)
        assert dt < 0.3, f"planner took {dt:.3f}s on {key}/{g.name}"


def test_random_tiny_groups_match_oracle(dbuf_lib, oracle_lib):
    rng = random.Random(2024)
    for _ in range(10000):
        specs = random_tiny_group(rng, max_tensors=6, max_rows=12, max_cols=5)
        m = rng.randint(1, 6)
        align = rng.choice([1, 1, 2, 4, 8])
        units = [rng.randint(1, 4) for _ in range(m)] if rng.random() < 0.3 else None
        q = _cplan(dbuf_lib, specs, m, units, align)
        o = oracle_lib.plan_specs(specs, m, units, align)
        assert (q["S"], q["offsets"]) == (o.S, [int(x) for x in o.offsets]), (specs, m, units, align)


def test_random_large_unit_groups_match_oracle(dbuf_lib, oracle_lib):
    """Tensors much larger than a shard with large units: exercises the jump over
    sizes that a tensor containing whole shards rules out."""
    rng = random.Random(31)
    for _ in range(300):
        specs = []
        for i in range(rng.randint(1, 7)):
            if rng.random() < 0.75:
                r = rng.choice([64, 128, 256, 384, 512, 1024])
                c = rng.choice([16, 48, 64, 96, 128, 176])
                specs.append(TensorSpec(f"m{i}", r, c, rng.choice([8, 16, 32, 64, 0])))
            else:
                specs.append(TensorSpec(f"v{i}", rng.randint(1, 500), 1, 1))
        m = rng.choice([2, 4, 8, 16, 32, 64])
        align = rng.choice([1, 4, 16])
        q = _cplan(dbuf_lib, specs, m, None, align)
        o = oracle_lib.plan_specs(specs, m, None, align)
        assert (q["S"], q["offsets"]) == (o.S, [int(x) for x in o.offsets]), (specs, m, align)


def test_empty_group_and_empty_tensors(dbuf_lib, oracle_lib):
    q = _cplan(dbuf_lib, [], 4)
    assert q["S"] == 0 and q["total"] == 0
    specs = [TensorSpec("a", 0, 5, 1), TensorSpec("b", 10, 1, 1), TensorSpec("c", 0, 1, 0)]
    q = _cplan(dbuf_lib, specs, 3, None, 4)
    o = oracle_lib.plan_specs(specs, 3, None, 4)
    assert (q["S"], q["offsets"]) == (o.S, [int(x) for x in o.offsets])
