"""GPU parity of the whole-matrix gather and scatter (dbuf_gather /
dbuf_scatter) against the oracle, bit for bit: m separate shard buffers, fp32
and bf16, uneven local_units, tensors spanning several shards, skipped
tensors, unaligned shard buffers (the element path), 1024 shards (a tensor
over ~960 of them); and at full size (a 7B
layer over 64 shards) the property that holds at any size: with the shards
cut from one flat buffer, each gathered matrix is the tensor's flat range and
a scattered matrix lands there."""
import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import TensorSpec

pytestmark = pytest.mark.gpu
DEV = "cuda"

SPECS = [TensorSpec("a", 300, 7, 1), TensorSpec("b", 0, 5, 1), TensorSpec("c", 1000, 3, 10),
         TensorSpec("d", 33, 1, 1), TensorSpec("e", 64, 64, 16), TensorSpec("big", 40000, 4, 1)]


def _np_dtype(dt):
    return np.float32 if dt == torch.float32 else np.uint16


def _to_dev(x: np.ndarray, dt, shift=0):
    t = torch.zeros(x.size + 8, dtype=dt, device=DEV)
    v = t[shift:shift + x.size]
    v.copy_(torch.from_numpy(x.view(np.int16) if dt == torch.bfloat16 else x).view(dt))
    return v


def _host(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu()
    return a.view(torch.int16).numpy().view(np.uint16) if a.dtype == torch.bfloat16 else a.numpy()


# A whole-matrix block of 50,000 elements forces S up to the block: with m=16
# most shard slices are empty.
SPECS_WHOLE = [TensorSpec("w", 200, 250, 200), TensorSpec("v", 100, 1, 1),
               TensorSpec("e", 64, 64, 16), TensorSpec("z", 0, 8, 1)]


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("which,m,units,shift", [("mixed", 4, None, 0), ("mixed", 7, None, 1),
                                                 ("mixed", 5, [1, 3, 2, 1, 4], 0),
                                                 ("whole", 16, None, 0), ("mixed", 1024, None, 0)])
def test_gather_scatter_match_oracle(dbuf_lib, oracle_lib, dt, which, m, units, shift):
    from fsdp_infra_gb300 import DBuffer
    SPECS_ = SPECS if which == "mixed" else SPECS_WHOLE
    rng = np.random.default_rng(m + shift)
    op = oracle_lib.plan_specs(SPECS_, m, units, 16)
    db = DBuffer(SPECS_, m, units, 16).upload()
    if which == "whole":  # all tensor data in the first two slices, the other 14 only padding
        assert db.S >= 50000
        assert max(o + s.numel for o, s in zip(db.offsets, SPECS_)) <= 2 * db.S
    assert db.offsets == [int(x) for x in op.offsets]
    npdt = _np_dtype(dt)
    hs = [rng.integers(0, 2 ** 15, n).astype(npdt) for n in db.shard_sizes()]
    shards = [_to_dev(h, dt, shift) for h in hs]
    # gather every other tensor; the rest must stay as filled
    hd = [None if t % 2 else np.full(s.numel, 3, npdt) for t, s in enumerate(SPECS_)]
    dd = [None if x is None else _to_dev(x, dt, shift) for x in hd]
    db.gather(shards, dd)
    oracle_lib.gather(op, hs, hd)
    torch.cuda.synchronize()
    for t in range(len(SPECS_)):
        if hd[t] is not None:
            assert np.array_equal(_host(dd[t]), hd[t]), f"gather t{t}"
    # scatter new matrices for the odd tensors
    hsrc = [None if t % 2 == 0 else rng.integers(0, 2 ** 15, s.numel).astype(npdt)
            for t, s in enumerate(SPECS_)]
    dsrc = [None if x is None else _to_dev(x, dt, shift) for x in hsrc]
    db.scatter(dsrc, shards)
    oracle_lib.scatter(op, hsrc, hs)
    torch.cuda.synchronize()
    for k in range(m):
        assert np.array_equal(_host(shards[k]), hs[k]), f"shard {k}"


def test_gather_scatter_full_size_dense7b_layer(dbuf_lib):
    from fsdp_infra_gb300 import DBuffer
    w = workload("dense7b")
    specs = w.groups[0].tensors
    db = DBuffer(specs, w.m, None, w.align).upload()
    gen = torch.Generator(device=DEV).manual_seed(5)
    flat = torch.empty(db.total, dtype=torch.float32, device=DEV)
    flat.normal_(generator=gen)
    b = db.shard_bounds
    shards = [flat[b[k]:b[k + 1]] for k in range(db.m)]
    mats = [torch.empty(s.numel, dtype=torch.float32, device=DEV) for s in specs]
    db.gather(shards, mats)
    for t, s in enumerate(specs):
        o = db.offsets[t]
        assert torch.equal(mats[t], flat[o:o + s.numel]), f"tensor {t}"
    before = flat.clone()
    new = [x * 2.0 + 1.0 for x in mats]
    db.scatter(new, shards)
    want = before.clone()
    for t, s in enumerate(specs):
        o = db.offsets[t]
        want[o:o + s.numel] = new[t]
    assert torch.equal(flat, want)
