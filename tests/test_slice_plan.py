"""Slice plans (dbuf_plan_slice): shard k of a planned group as a rank's local
buffer, host side (no GPU).

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer: every
rank owns one slice [B_k, B_{k+1}) of the global buffer; §4 and §6.3: no block
crosses a shard, so each rank's operators (and its block quantisation) need
only its slice.  The expected pieces are computed here from the oracle's
layout: tensor t's piece in slice k is [l_t, l_t + n_t) intersected with
[B_k, B_{k+1}); a quantised tensor's blocks in the slice are its block rows
whose first element lies inside the slice.
"""
import random

import pytest

from workloads import workload
from workloads.configs import TensorSpec


def _random_group(rng):
    specs = []
    for i in range(rng.randint(1, 10)):
        kind = rng.random()
        if kind < 0.2:
            specs.append(TensorSpec(f"v{i}", rng.randint(0, 300), 1, 1))
        elif kind < 0.45:
            r, c = rng.randint(1, 40), rng.choice([4, 8, 12, 16, 20])
            specs.append(TensorSpec(f"m{i}", r, c, rng.choice([0, 1, 2, 3])))
        elif kind < 0.8:
            qr, qc = rng.choice([(4, 4), (2, 8), (1, 8), (8, 4), (3, 4)])
            r, c = rng.randint(1, 30), rng.choice([8, 12, 16, 24])
            gran = qr * rng.randint(1, 3)
            specs.append(TensorSpec(f"q{i}", r, c, gran, (qr, qc), rng.choice(["e4m3", "int8"])))
        else:
            r, c = rng.randint(1, 20), rng.choice([4, 8])
            specs.append(TensorSpec(f"w{i}", r, c, 0, (0, 0), "int8"))
    return specs


def _expected(op, specs, k):
    """Pieces, local offsets and block-scale range of slice k from the oracle's layout."""
    B0, B1 = int(op.bounds[k]), int(op.bounds[k + 1])
    src, num, local = [], [], []
    scale_before, scale_in = 0, 0
    for t, s in enumerate(specs):
        l, n = int(op.offsets[t]), s.numel
        lo, hi = max(l, B0), min(l + n, B1)
        if hi > lo:
            src.append(lo - l)
            num.append(hi - lo)
            local.append(lo - B0)
        else:
            num.append(0)
            src.append(None)
            local.append(None)
        if s.quant and n:
            qr = s.qblock[0] or s.rows
            qc = s.qblock[1] or s.cols
            nbc = -(-s.cols // qc)
            for bi in range(-(-s.rows // qr)):
                first = l + bi * qr * s.cols
                if first < B0:
                    scale_before += nbc
                elif first < B1:
                    scale_in += nbc
    return {"len": B1 - B0, "src": src, "num": num, "local": local,
            "scale_base": scale_before, "n_scales": scale_in}


def _check_slices(dbuf, oracle_lib, specs, m, units, align):
    from fsdp_infra_gb300 import DBuffer
    op = oracle_lib.plan_specs(specs, m, units, align)
    db = DBuffer(specs, m, units, align)
    assert db.offsets == [int(x) for x in op.offsets]
    n_scales = 0
    for k in range(m):
        sl = db.slice(k)
        want = _expected(op, specs, k)
        assert sl.slice_k == k and sl.global_offset == int(op.bounds[k])
        assert sl.total == want["len"] and sl.S == want["len"]
        assert sl.shard_bounds == [0, want["len"]]
        assert sl.piece_numels == want["num"]
        for t in range(len(specs)):
            if want["num"][t]:
                assert sl.src_offsets[t] == want["src"][t], (k, t)
                assert sl.offsets[t] == want["local"][t], (k, t)
                assert 0 <= sl.offsets[t] and sl.offsets[t] + want["num"][t] <= sl.total
                assert sl.offsets[t] % align == 0
        assert sl.scale_base == want["scale_base"] and sl.n_scales == want["n_scales"], k
        assert sl.scale_base == n_scales  # the slices' scales tile the full range in order
        n_scales += sl.n_scales
        # the local scale numbering of a piece: its first block row's index in the
        # full numbering, minus the slice's base
        for t, s in enumerate(specs):
            if s.quant and want["num"][t]:
                qr = s.qblock[0] or s.rows
                qc = s.qblock[1] or s.cols
                nbc = -(-s.cols // qc)
                first_row = want["src"][t] // s.cols
                assert first_row % qr == 0
                glob = db.scale_offsets[t] + first_row // qr * nbc
                assert sl.scale_offsets[t] == glob - sl.scale_base, (k, t)
        assert dbuf.dbuf_workspace_bytes(sl.handle, dbuf.DBUF_OP_NORM_NONFINITE) > 0
        sl.close()
    assert n_scales == db.n_scales
    db.close()


@pytest.mark.parametrize("seed", range(5))
def test_slices_of_random_groups(dbuf_lib, oracle_lib, seed):
    rng = random.Random(900 + seed)
    for _ in range(25):
        specs = _random_group(rng)
        m = rng.randint(1, 6)
        units = [rng.randint(1, 3) for _ in range(m)] if rng.random() < 0.4 else None
        align = rng.choice([1, 4, 16])
        _check_slices(dbuf_lib, oracle_lib, specs, m, units, align)


@pytest.mark.parametrize("key", ["tiny", "llama_layer", "moe"])
def test_slices_of_workloads(dbuf_lib, oracle_lib, key):
    w = workload(key)
    _check_slices(dbuf_lib, oracle_lib, w.groups[0].tensors, w.m, w.local_units, w.align)


def test_slice_errors(dbuf_lib):
    d = dbuf_lib
    p = d.dbuf_plan([(8, 8, 1), (16, 1, 1)], 3)
    try:
        for k in (-1, 3, 100):
            with pytest.raises(d.DbufError) as e:
                d.dbuf_plan_slice(p, k)
            assert e.value.code == d.DBUF_EINVAL
        s = d.dbuf_plan_slice(p, 1)
        try:
            with pytest.raises(d.DbufError) as e:  # a slice of a slice
                d.dbuf_plan_slice(s, 0)
            assert e.value.code == d.DBUF_EINVAL
            with pytest.raises(d.DbufError) as e:  # a full plan has no slice info
                d.dbuf_plan_slice_info(p, 2)
            assert e.value.code == d.DBUF_EINVAL
            with pytest.raises(d.DbufError) as e:  # gather needs every shard
                d.dbuf_gather(s, 0, d.DBUF_F32, 0)
            assert e.value.code == d.DBUF_EINVAL
        finally:
            d.dbuf_plan_free(s)
    finally:
        d.dbuf_plan_free(p)
