"""Pins of the oracle's whole-matrix gather and scatter (no GPU).

Independent of the oracle's shard lookup: when the m shard buffers are the
consecutive slices [B_k, B_{k+1}) of one flat buffer, gathering tensor t must
give exactly the flat range [l_t, l_t + n_t); scattering matrices back must
change only those ranges (padding untouched) and invert the gather; skipped
tensors are neither read nor written.  Covers tensors spanning three or more
shards, uneven local_units, empty tensors, fp32 and bf16 bit patterns.
"""
import numpy as np
import pytest

from workloads.configs import TensorSpec


def _specs():
    return [TensorSpec("a", 300, 7, 1), TensorSpec("b", 0, 5, 1), TensorSpec("c", 1000, 3, 10),
            TensorSpec("d", 33, 1, 1), TensorSpec("e", 64, 64, 16), TensorSpec("big", 4000, 4, 1)]


def _split(flat, bounds):
    return [flat[int(bounds[k]):int(bounds[k + 1])].copy() for k in range(len(bounds) - 1)]


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
@pytest.mark.parametrize("m,units", [(4, None), (7, None), (5, [1, 3, 2, 1, 4])])
def test_gather_is_the_flat_range(oracle_lib, dtype, m, units):
    rng = np.random.default_rng(m)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, m, units, 16)
    flat = rng.integers(0, 2 ** 16, p.total).astype(dtype)
    shards = _split(flat, p.bounds)
    dsts = [np.full(s.numel, 7, dtype) for s in specs]
    oracle_lib.gather(p, shards, dsts)
    spans = 0
    for t, s in enumerate(specs):
        o = int(p.offsets[t])
        assert np.array_equal(dsts[t], flat[o:o + s.numel])
        ks = {int(np.searchsorted(p.bounds, x, side="right")) - 1 for x in range(o, o + s.numel)}
        spans = max(spans, len(ks))
    assert spans >= 3          # some tensor is assembled from three or more shards


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_scatter_changes_only_tensor_ranges_and_inverts_gather(oracle_lib, dtype):
    rng = np.random.default_rng(1)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, 6, None, 16)
    flat = rng.integers(0, 2 ** 16, p.total).astype(dtype)
    shards = _split(flat, p.bounds)
    new = [rng.integers(0, 2 ** 16, s.numel).astype(dtype) for s in specs]
    oracle_lib.scatter(p, new, shards)
    want = flat.copy()
    for t, s in enumerate(specs):
        o = int(p.offsets[t])
        want[o:o + s.numel] = new[t]
    assert np.array_equal(np.concatenate(shards), want)
    back = [np.zeros(s.numel, dtype) for s in specs]
    oracle_lib.gather(p, shards, back)
    for t in range(len(specs)):
        assert np.array_equal(back[t], new[t])


def test_skipped_tensors(oracle_lib):
    rng = np.random.default_rng(2)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, 3, None, 16)
    flat = rng.standard_normal(p.total).astype(np.float32)
    shards = _split(flat, p.bounds)
    dsts = [None if t % 2 else np.zeros(s.numel, np.float32) for t, s in enumerate(specs)]
    oracle_lib.gather(p, shards, dsts)
    srcs = [None if t % 2 == 0 else np.ones(s.numel, np.float32) for t, s in enumerate(specs)]
    before = [x.copy() for x in shards]
    oracle_lib.scatter(p, srcs, shards)
    got = np.concatenate(shards)
    ref = np.concatenate(before)
    for t, s in enumerate(specs):
        o = int(p.offsets[t])
        if srcs[t] is None:
            assert np.array_equal(got[o:o + s.numel], ref[o:o + s.numel])
        else:
            assert np.all(got[o:o + s.numel] == 1.0)
