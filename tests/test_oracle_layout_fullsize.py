"""The oracle planner at the workloads' full sizes, against a literal scan.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 Planning
algorithm (problem formulation): at a fixed per-shard size S the canonical
layout places each tensor at the smallest aligned start after the previous
tensor that keeps every shard boundary inside it a whole number of units from
its start.  The oracle finds that start with a per-shard jump (the pages'
3-case analysis); ``layout_check.literal_greedy`` finds it by examining every
aligned candidate in order.  The two share no code.

Checked on all five workloads (the 7B layer at S* = 23,592,960 and the
2000-tensor group included):
- at the oracle's S* the literal scan returns the oracle's offsets exactly;
- at S* - a the literal scan finds no layout;
- minimality: every aligned size in [LB, S*) has no layout for the tiny and
  MoE groups (16 candidates each), and a seeded sample of sizes has none for the
  others.  The greedy placement is exact at a fixed size (pinned against the
  assumption-free brute force on small groups), so a size the literal greedy
  rejects admits no layout at all;
- complete minimality for the 7B layer and the embedding (1.28M and 3K
  candidate sizes): a tensor longer than 2S holds two consecutive boundaries,
  so (iii) makes its unit divide S (``two_boundary_survivors``, itself checked
  against the brute force on small even groups); that rules out every size
  below S* but a few, and the literal scan rejects those.
"""
import random

import numpy as np
import pytest

from workloads import workload, WORKLOADS

from layout_check import (brute_force_plan, check_layout, feasible_placement, literal_greedy,
                          two_boundary_survivors, unit_of)
from workloads.configs import TensorSpec

CASES = [(key, gi) for key in WORKLOADS for gi in range(len(workload(key).groups))]

# sampled sizes below S* per group (None = every size); the 7B layer's
# rejections scan the whole 1.5e9-element buffer (about 4 s each)
SAMPLES = {("dense7b", 0): 1, ("dense7b", 1): 32, ("llama_layer", 0): 64, ("mixed", 0): 32,
           ("tiny", 0): None, ("moe", 0): None}


def _lower_bound(w, g):
    units = w.local_units or [1] * w.m
    big = max(min(unit_of(s.rows, s.cols, s.gran_rows), s.numel) for s in g.tensors)
    lb = max(-(-g.numel // sum(units)), -(-big // max(units)))
    return -(-lb // w.align) * w.align


@pytest.mark.parametrize("key,gi", CASES)
def test_literal_scan_gives_the_oracle_layout(oracle_plans, key, gi):
    w = workload(key)
    g = w.groups[gi]
    p = oracle_plans(key, gi)
    offs = literal_greedy(g.tensors, p.S, w.m, w.local_units, w.align)
    assert offs == [int(x) for x in p.offsets], (key, gi)
    assert not check_layout(g.tensors, offs, p.bounds, w.align)
    if p.S - w.align >= _lower_bound(w, g):
        assert literal_greedy(g.tensors, p.S - w.align, w.m, w.local_units, w.align) is None


@pytest.mark.parametrize("key,gi", CASES)
def test_no_smaller_size_has_a_layout(oracle_plans, key, gi):
    w = workload(key)
    g = w.groups[gi]
    p = oracle_plans(key, gi)
    lb = _lower_bound(w, g)
    sizes = list(range(lb, p.S, w.align))
    k = SAMPLES[(key, gi)]
    if k is not None and len(sizes) > k:
        sizes = random.Random(11 + gi).sample(sizes, k)
    for S in sizes:
        assert literal_greedy(g.tensors, S, w.m, w.local_units, w.align) is None, (key, gi, S)


@pytest.mark.parametrize("seed", range(4))
def test_two_boundary_lemma_keeps_every_feasible_size(seed):
    """On small even groups with row units, every size at which the
    assumption-free brute force finds a layout survives the lemma, and the
    lemma does reject sizes (it is not vacuous on these groups)."""
    rng = random.Random(500 + seed)
    rejected = 0
    for _ in range(25):
        specs = []
        for i in range(rng.randint(1, 4)):
            rows, cols = rng.randint(1, 12), rng.randint(1, 3)
            specs.append(TensorSpec(f"t{i}", rows, cols, rng.choice([0, 1, 2, 3])))
        m = rng.randint(2, 5)
        E = sum(t.numel for t in specs)
        U, _ = brute_force_plan(specs, m, None, 1)
        sizes = list(range(1, U + 2 * E + 2))
        keep = set(int(x) for x in two_boundary_survivors(specs, sizes))
        rejected += len(sizes) - len(keep)
        for S in sizes:
            if feasible_placement(specs, S, m, None, 1) is not None:
                assert S in keep, (specs, m, S)
    assert rejected > 0


@pytest.mark.parametrize("gi", [0, 1])
def test_dense7b_minimality_is_complete(oracle_plans, gi):
    w = workload("dense7b")
    g = w.groups[gi]
    p = oracle_plans("dense7b", gi)
    sizes = np.arange(_lower_bound(w, g), p.S, w.align, dtype=np.int64)
    left = two_boundary_survivors(g.tensors, sizes)
    assert len(left) <= 64, len(left)
    for S in left:
        assert literal_greedy(g.tensors, int(S), w.m, w.local_units, w.align) is None, (gi, S)
