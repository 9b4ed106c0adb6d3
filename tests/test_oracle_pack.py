"""Pins of the oracle's copy-in (pack) and copy-out (unpack), independent of it.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer and
Figure 2: copy-in writes every tensor into its range of the flat buffer and
copy-out reads it back; padding between tensors is never written.  "PyTorch
FSDP: Experiences on Scaling Fully Sharded Data Parallel", native mixed
precision: the fp32 master copy is cast to bf16 once per flat parameter.

Pins:
- a hand-worked three-tensor plan whose whole expected buffer, padding included,
  is written out with its derivation (tests/golden/pack_hand_worked.json), in
  fp32 and in bf16 with rounding-critical values;
- bitwise round-trip identity (pack then unpack returns the inputs) for f32->f32
  and bf16->bf16 on random multi-tensor plans, with padding sentinels that must
  survive, NaN payloads and arbitrary 16-bit patterns included;
- pack f32->bf16 followed by unpack bf16->f32 equal to torch's CPU
  float32 -> bfloat16 -> float32 conversion element by element;
- planted mistakes (an offset one element early, one element too many copied)
  each fail one of the checks above.
"""
import ctypes
import json
import os
import random

import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pack_hand_worked.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _specs(case):
    return [TensorSpec(f"t{i}", r, c, g) for i, (r, c, g) in enumerate(case["tensors"])]


def _bits32(hexes):
    return np.array([int(h, 16) for h in hexes], np.uint32)


def test_hand_worked_plan(oracle_lib):
    case = _golden()
    p = oracle_lib.plan_specs(_specs(case), case["m"], None, case["align"])
    assert p.S == case["S"]
    assert list(map(int, p.offsets)) == case["offsets"]
    assert list(map(int, p.bounds)) == case["bounds"]


def test_hand_worked_pack_f32(oracle_lib):
    case = _golden()
    g = case["f32"]
    p = oracle_lib.plan_specs(_specs(case), case["m"], None, case["align"])
    sentinel = np.array([int(g["padding_sentinel_bits"], 16)], np.uint32).view(np.float32)[0]
    buf = np.full(p.total, sentinel, np.float32)
    srcs = [np.array(x, np.float32) for x in g["inputs"]]
    oracle_lib.pack(p, srcs, buf)
    want = np.array(g["buffer"], np.float32)
    assert np.array_equal(buf.view(np.uint32), want.view(np.uint32))
    dsts = [np.zeros_like(s) for s in srcs]
    oracle_lib.unpack(p, buf, dsts)
    for s, d in zip(srcs, dsts):
        assert np.array_equal(s.view(np.uint32), d.view(np.uint32))


def test_hand_worked_pack_bf16(oracle_lib):
    case = _golden()
    g = case["bf16"]
    p = oracle_lib.plan_specs(_specs(case), case["m"], None, case["align"])
    buf = np.full(p.total, int(g["padding_sentinel_bits"], 16), np.uint16)
    srcs = [_bits32(x).view(np.float32) for x in g["input_bits"]]
    oracle_lib.pack(p, srcs, buf)
    want = np.array([int(h, 16) for h in g["buffer_bits"]], np.uint16)
    assert np.array_equal(buf, want)
    # the hand derivation agrees with torch's conversion (a library routine)
    for t, s in enumerate(srcs):
        o = case["offsets"][t]
        tb = torch.from_numpy(s.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(tb, want[o:o + s.size])
    # unpack bf16 -> fp32 is exact: the pattern shifted up by 16 bits
    dsts = [np.zeros(s.size, np.float32) for s in srcs]
    oracle_lib.unpack(p, buf, dsts)
    for t, d in enumerate(dsts):
        o = case["offsets"][t]
        assert np.array_equal(d.view(np.uint32), want[o:o + d.size].astype(np.uint32) << 16)


def _random_group(rng):
    specs = []
    for i in range(rng.randint(1, 9)):
        kind = rng.random()
        if kind < 0.25:
            specs.append(TensorSpec(f"v{i}", rng.randint(0, 70), 1, 1))
        elif kind < 0.6:
            r, c = rng.randint(1, 24), rng.randint(1, 9)
            specs.append(TensorSpec(f"m{i}", r, c, rng.choice([0, 1, 2, 3, 8])))
        else:
            r, c = rng.randint(1, 12), rng.randint(1, 5)
            specs.append(TensorSpec(f"w{i}", r, c, 0))
    return specs


def _random_plan(oracle_lib, rng):
    specs = _random_group(rng)
    m = rng.randint(1, 7)
    units = [rng.randint(1, 4) for _ in range(m)] if rng.random() < 0.4 else None
    align = rng.choice([1, 2, 4, 16])
    return specs, oracle_lib.plan_specs(specs, m, units, align)


def _padding(p, specs):
    mask = np.ones(p.total, bool)
    for o, s in zip(p.offsets, specs):
        mask[int(o):int(o) + s.numel] = False
    return mask


@pytest.mark.parametrize("seed", range(4))
def test_round_trip_f32_bitwise(oracle_lib, seed):
    rng = random.Random(300 + seed)
    nrng = np.random.default_rng(300 + seed)
    for _ in range(60):
        specs, p = _random_plan(oracle_lib, rng)
        # arbitrary bit patterns: NaN payloads, infinities, subnormals, -0
        srcs = [nrng.integers(0, 2 ** 32, s.numel, dtype=np.uint64).astype(np.uint32)
                .view(np.float32) for s in specs]
        sentinel = np.uint32(0x7FC0BEEF).view(np.float32)
        buf = np.full(p.total, sentinel, np.float32)
        oracle_lib.pack(p, srcs, buf)
        pad = _padding(p, specs)
        assert np.all(buf.view(np.uint32)[pad] == 0x7FC0BEEF)
        dsts = [np.full(s.numel, 1.5, np.float32) for s in specs]
        oracle_lib.unpack(p, buf, dsts)
        for s, d in zip(srcs, dsts):
            assert np.array_equal(s.view(np.uint32), d.view(np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_round_trip_bf16_bitwise(oracle_lib, seed):
    rng = random.Random(400 + seed)
    nrng = np.random.default_rng(400 + seed)
    for _ in range(60):
        specs, p = _random_plan(oracle_lib, rng)
        srcs = [nrng.integers(0, 2 ** 16, s.numel, dtype=np.uint32).astype(np.uint16)
                for s in specs]
        buf = np.full(p.total, 0xA5A5, np.uint16)
        oracle_lib.pack(p, srcs, buf)
        assert np.all(buf[_padding(p, specs)] == 0xA5A5)
        dsts = [np.zeros(s.numel, np.uint16) for s in specs]
        oracle_lib.unpack(p, buf, dsts)
        for s, d in zip(srcs, dsts):
            assert np.array_equal(s, d)


@pytest.mark.parametrize("seed", range(3))
def test_pack_cast_then_unpack_is_torch_bf16_rounding(oracle_lib, seed):
    rng = random.Random(500 + seed)
    nrng = np.random.default_rng(500 + seed)
    for _ in range(40):
        specs, p = _random_plan(oracle_lib, rng)
        srcs = []
        for s in specs:
            x = nrng.integers(0, 2 ** 32, s.numel, dtype=np.uint64).astype(np.uint32)
            # half of them on the rounding-critical low halves
            lows = nrng.choice(np.array([0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32),
                               s.numel)
            pick = nrng.random(s.numel) < 0.5
            x[pick] = (x[pick] & 0xFFFF0000) | lows[pick]
            srcs.append(x.view(np.float32))
        buf = np.full(p.total, 0x5A5A, np.uint16)
        oracle_lib.pack(p, srcs, buf)
        assert np.all(buf[_padding(p, specs)] == 0x5A5A)
        dsts = [np.zeros(s.numel, np.float32) for s in specs]
        oracle_lib.unpack(p, buf, dsts)
        for s, d in zip(srcs, dsts):
            want = torch.from_numpy(s.copy()).to(torch.bfloat16).to(torch.float32).numpy()
            nan = np.isnan(s)
            assert np.array_equal(d.view(np.uint32)[~nan], want.view(np.uint32)[~nan])
            assert np.all(np.isnan(d[nan]))
            assert np.array_equal(np.signbit(d[nan]), np.signbit(s[nan]))
            # and equal to the oracle's own pinned encoder, element by element
            enc = oracle_lib.f32_to_bf16_bits(s).astype(np.uint32) << 16
            assert np.array_equal(d.view(np.uint32), enc)


def _raw_pack(oracle_lib, offsets, numel, srcs, buf):
    """orc_pack with caller-chosen offsets and sizes (to plant mistakes)."""
    n = len(srcs)
    ptrs = (ctypes.c_void_p * n)(*[s.ctypes.data for s in srcs])
    off = np.ascontiguousarray(offsets, np.int64)
    num = np.ascontiguousarray(numel, np.int64)
    oracle_lib.lib().orc_pack(n, off.ctypes.data_as(ctypes.c_void_p),
                              num.ctypes.data_as(ctypes.c_void_p), ptrs, oracle_lib.F32,
                              buf.ctypes.data_as(ctypes.c_void_p), oracle_lib.F32)


def test_planted_mistakes_fail_the_checks(oracle_lib):
    """An offset one element early overwrites the previous tensor's last element
    (round trip fails); one element too many writes into padding (sentinel
    check fails).  The checks above would catch both in the oracle."""
    case = _golden()
    specs = _specs(case)
    p = oracle_lib.plan_specs(specs, case["m"], None, case["align"])
    srcs = [np.array(x, np.float32) for x in case["f32"]["inputs"]]
    numel = [s.numel for s in specs]

    early = [int(o) for o in p.offsets]
    early[1] -= 1
    buf = np.full(p.total, 7777.0, np.float32)
    _raw_pack(oracle_lib, early, numel, srcs, buf)
    dsts = [np.zeros_like(s) for s in srcs]
    oracle_lib.unpack(p, buf, dsts)
    assert not np.array_equal(dsts[0], srcs[0])

    longer = list(numel)
    longer[2] += 1
    buf = np.full(p.total, 7777.0, np.float32)
    grown = [srcs[0], srcs[1], np.append(srcs[2], np.float32(9.0))]
    _raw_pack(oracle_lib, p.offsets, longer, grown, buf)
    assert not np.all(buf[_padding(p, specs)] == 7777.0)
