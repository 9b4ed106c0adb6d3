"""Placement orders (default, block size, shape): the library's dbuf_order
equals the oracle's, and the oracle's orders are pinned by their defining
properties (a permutation; keys non-increasing; equal keys keep the given
order) -- host only, no GPU."""
import random

import pytest

from workloads import WORKLOADS, workload
from workloads.configs import TensorSpec, random_tiny_group


def _check_order(specs, perm, key):
    assert sorted(perm) == list(range(len(specs)))
    keys = [key(specs[t]) for t in perm]
    assert all(keys[i] >= keys[i + 1] for i in range(len(keys) - 1))
    for i in range(len(perm) - 1):
        if keys[i] == keys[i + 1]:
            assert perm[i] < perm[i + 1]          # stable


def test_oracle_orders_by_definition(oracle_lib):
    rng = random.Random(0)
    for _ in range(50):
        specs = [TensorSpec(f"t{i}", rng.choice([0, 1, 3, 64, 128]), rng.choice([1, 4, 64]),
                            rng.choice([0, 1, 16, 128])) for i in range(rng.randint(0, 30))]
        assert oracle_lib.order(specs, "default") == list(range(len(specs)))
        _check_order(specs, oracle_lib.order(specs, "block"), oracle_lib.shard_unit)
        _check_order(specs, oracle_lib.order(specs, "shape"), lambda s: (s.rows, s.cols))
    # a hand-made case: g = 128*64, 16*4, 4*1 (whole tensor), 32*64 (gran >= rows)
    specs = [TensorSpec("a", 256, 64, 128), TensorSpec("b", 64, 4, 16), TensorSpec("c", 4, 1, 0),
             TensorSpec("d", 32, 64, 64)]
    assert oracle_lib.order(specs, "block") == [0, 3, 1, 2]
    assert oracle_lib.order(specs, "shape") == [0, 1, 3, 2]


@pytest.mark.parametrize("kind", ["default", "block", "shape"])
def test_library_orders_match_oracle(dbuf_lib, oracle_lib, kind):
    rng = random.Random(1)
    groups = [g.tensors for key in WORKLOADS for g in workload(key).groups]
    groups += [random_tiny_group(rng) for _ in range(20)]
    for specs in groups:
        assert dbuf_lib.dbuf_order(list(specs), kind) == oracle_lib.order(list(specs), kind)


def test_order_rejects_unknown_kind(dbuf_lib):
    import ctypes
    arr = dbuf_lib._spec_array([TensorSpec("a", 4, 4, 1)])
    perm = (ctypes.c_int32 * 1)()
    assert dbuf_lib.library().dbuf_order(arr, 1, 7, perm) == dbuf_lib.DBUF_EINVAL
