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
  rejects admits no layout at all.
"""
import random

import pytest

from workloads import workload, WORKLOADS

from layout_check import check_layout, literal_greedy, unit_of

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
