"""GPU parity of the 8-bit AdamW step (dbuf_adamw8_step) against the oracle.

Bit-exact: parameters, both code arrays (the whole buffers, so bytes outside
quantised tensors must stay as they were), both scale arrays and the compact
fp32 moments, over several steps with clipping and a skipped step.  Covered:
square 32x32 blocks (one warp per block, moments in registers), 1x128 row
blocks (4 lanes per block), whole-row and 128x128 blocks (the recompute pass),
ragged edge blocks, odd widths and unaligned buffers (the scalar path), tiny
values (the IEEE-division path of the quotient), all-zero blocks, and one
full-size 7B-shaped layer with 32x32 blocks.
"""
import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import TensorSpec, adam8_group, grad_values, param_values

from gpu_helpers import assert_bits_equal, f32

pytestmark = pytest.mark.gpu

DEV = "cuda"
HP = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)

SPECS = [
    TensorSpec("w_sq", 70, 96, 32, qblock=(32, 32), quant="int8"),
    TensorSpec("bias", 57, 1, 1),
    TensorSpec("w_row", 33, 130, 1, qblock=(1, 128), quant="e4m3"),
    TensorSpec("empty", 0, 64, 32, qblock=(32, 32), quant="int8"),
    TensorSpec("w_odd", 15, 7, 5, qblock=(5, 3), quant="int8"),
    TensorSpec("norm", 96, 1, 0, kind="norm"),
    TensorSpec("w_full", 8, 40, 8, qblock=(8, 0), quant="int8"),
    TensorSpec("w_rows", 64, 256, 1, qblock=(1, 128), quant="int8"),
    TensorSpec("w_big", 256, 136, 128, qblock=(128, 128), quant="e4m3"),
    TensorSpec("w_tiny", 64, 64, 32, qblock=(32, 32), quant="int8"),     # tiny values
]


def _db(specs, m, units=None, align=16):
    from fsdp_infra_gb300 import DBuffer
    return DBuffer(specs, m, units, align).upload()


def _dev(x: np.ndarray, shift: int = 0) -> torch.Tensor:
    """Device copy of x, optionally at an element offset inside a larger
    allocation (to take the unaligned paths)."""
    t = torch.zeros(x.size + 8, dtype=torch.from_numpy(x[:0]).dtype, device=DEV)
    v = t[shift:shift + x.size]
    v.copy_(torch.from_numpy(x))
    return v


class Case:
    def __init__(self, oracle_lib, specs, m, units=None, align=16, seed=0, zero=False, shift=0):
        self.specs, self.ol = specs, oracle_lib
        self.op = oracle_lib.plan_specs(specs, m, units, align)
        self.db = _db(specs, m, units, align)
        assert self.db.offsets == [int(x) for x in self.op.offsets]
        so, n_state = oracle_lib.state_offsets(specs)
        assert self.db.state_offsets == [int(x) for x in so] and self.db.n_state == n_state
        self.rng = np.random.default_rng(seed)
        tot, ns = self.op.total, max(self.db.n_scales, 1)
        self.h = {"p": np.zeros(tot, np.float32), "mc": np.zeros(tot, np.uint8),
                  "vc": np.zeros(tot, np.uint8), "ms": np.zeros(ns, np.float32),
                  "vs": np.zeros(ns, np.float32), "m32": np.zeros(max(n_state, 1), np.float32),
                  "v32": np.zeros(max(n_state, 1), np.float32)}
        self.h["p"][:] = self.rng.standard_normal(tot).astype(np.float32) * 0.02
        if not zero:
            self.h["mc"][:] = self.rng.integers(0, 256, tot).astype(np.uint8)
            self.h["vc"][:] = self.rng.integers(0, 256, tot).astype(np.uint8)
            self.h["ms"][:] = self.rng.uniform(1e-7, 1e-5, ns).astype(np.float32)
            self.h["vs"][:] = self.rng.uniform(1e-12, 1e-9, ns).astype(np.float32)
            self.h["m32"][:] = self.rng.standard_normal(self.h["m32"].size).astype(np.float32) * 1e-4
            self.h["v32"][:] = np.abs(self.rng.standard_normal(self.h["v32"].size)).astype(np.float32) * 1e-8
        self.shift = shift
        self.d = {k: _dev(v, shift if k in ("p", "mc", "vc") else 0) for k, v in self.h.items()}
        self.state = {"m_codes": self.d["mc"], "v_codes": self.d["vc"], "m_scales": self.d["ms"],
                      "v_scales": self.d["vs"], "m32": self.d["m32"], "v32": self.d["v32"]}
        self.norm = torch.zeros(1, dtype=torch.float32, device=DEV)
        self.flag = torch.zeros(1, dtype=torch.int32, device=DEV)

    def grad(self):
        g = (self.rng.standard_normal(self.op.total) * 1e-3).astype(np.float32)
        for s, o in zip(self.specs, self.op.offsets):
            if s.name == "w_tiny":
                g[int(o):int(o) + s.numel] *= np.float32(1e-26)
            if s.name == "w_sq":     # one all-zero block
                r = g[int(o):int(o) + s.numel].reshape(s.rows, s.cols)
                r[32:64, 32:64] = 0.0
            if s.name == "w_rows":   # zeros among normal values (mixed units)
                g[int(o):int(o) + s.numel:7] = 0.0
            if s.name == "b_zero":   # one whole 128x128 block of zero gradients
                r = g[int(o):int(o) + s.numel].reshape(s.rows, s.cols)
                r[128:256, 0:128] = 0.0
        return g

    def step(self, step, clip=False, skip=False, hp=None):
        hp = HP if hp is None else hp
        g = self.grad()
        gd = _dev(g, self.shift)
        _, wt, _ = self.ol.norm_nonfinite(self.op, g)
        total32 = float(np.float32(wt))
        self.norm.fill_(total32)
        self.flag.fill_(1 if skip else 0)
        max_norm = 0.5 * total32 if clip else 0.0
        self.db.adamw8_step(self.d["p"], gd, self.state, step=step, max_norm=max_norm,
                            total_norm=self.norm, nonfinite=self.flag, **hp)
        b1, b2 = hp["betas"]
        h = self.h
        self.ol.adamw8(self.op, self.specs, h["p"], g, h["mc"], h["vc"], h["ms"], h["vs"],
                       h["m32"], h["v32"], lr=hp["lr"], beta1=b1, beta2=b2, eps=hp["eps"],
                       weight_decay=hp["weight_decay"], step=step, max_norm=max_norm,
                       total_norm=total32, nonfinite=1 if skip else 0)
        torch.cuda.synchronize()
        for k in h:
            got = self.d[k].cpu().numpy()
            if got.dtype == np.uint8:
                bad = np.flatnonzero(got != h[k])
                assert bad.size == 0, f"{k} step {step}: {bad.size} codes differ, first at {bad[:5]}"
            else:
                assert_bits_equal(got, h[k], f"{k} step {step}")


def test_adamw8_mixed_shapes_steps(dbuf_lib, oracle_lib):
    c = Case(oracle_lib, SPECS, 3)
    for step, (clip, skip) in enumerate([(False, False), (True, False), (True, True),
                                         (False, False)], start=1):
        c.step(step, clip, skip)


def test_adamw8_zero_state_first_steps(dbuf_lib, oracle_lib):
    c = Case(oracle_lib, SPECS, 2, zero=True, seed=1)
    for step in (1, 2, 3):
        c.step(step, clip=True)


@pytest.mark.parametrize("m,align,shift", [(5, 1, 0), (2, 16, 1), (4, 16, 2)])
def test_adamw8_ragged_and_unaligned(dbuf_lib, oracle_lib, m, align, shift):
    c = Case(oracle_lib, SPECS, m, align=align, shift=shift, seed=2)
    c.step(1, clip=True)
    c.step(2)


def test_adamw8_uneven_units(dbuf_lib, oracle_lib):
    specs = [TensorSpec(f"e{i}", 96, 160, 1, qblock=(1, 128), quant="int8") for i in range(6)]
    specs.append(TensorSpec("router", 96, 12, 1, qblock=(1, 128), quant="int8"))
    c = Case(oracle_lib, specs, 4, units=[1, 3, 2, 4], seed=3)
    c.step(1)
    c.step(2, clip=True)


def test_adamw8_llama_layer_32x32(dbuf_lib, oracle_lib):
    g = adam8_group(workload("llama_layer").groups[0])
    c = Case(oracle_lib, list(g.tensors), 8, seed=4)
    c.step(5, clip=True)


def test_adamw8_dense7b_layer_full_size(dbuf_lib, oracle_lib):
    """One step on the full-size 7B-shaped layer with the 8-bit Adam blocks
    (32x32, 32-row granularity); each tensor checked against the oracle run on
    that tensor alone."""
    w = workload("dense7b")
    specs = list(adam8_group(w.groups[0]).tensors)
    db = _db(specs, w.m)
    gen = torch.Generator().manual_seed(7)
    params = [param_values(w, 0, t).reshape(-1).float() for t in range(len(specs))]
    grads = [grad_values(w, 0, t).reshape(-1).float() for t in range(len(specs))]
    p = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    g = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    st = db.new_adamw8_state()
    mc0 = torch.randint(0, 256, (db.total,), dtype=torch.uint8, generator=gen)
    vc0 = torch.randint(0, 256, (db.total,), dtype=torch.uint8, generator=gen)
    ms0 = torch.rand(max(db.n_scales, 1), generator=gen) * 1e-5
    vs0 = torch.rand(max(db.n_scales, 1), generator=gen) * 1e-9
    st["m_codes"].copy_(mc0); st["v_codes"].copy_(vc0)
    st["m_scales"].copy_(ms0); st["v_scales"].copy_(vs0)
    for t, s in enumerate(specs):
        o = db.offsets[t]
        p[o:o + s.numel].copy_(params[t])
        g[o:o + s.numel].copy_(grads[t])
    total = torch.tensor([0.75], device=DEV)
    db.adamw8_step(p, g, st, step=3, max_norm=0.5, total_norm=total, **HP)
    torch.cuda.synchronize()
    b1, b2 = HP["betas"]
    for t, s in enumerate(specs):
        sp = oracle_lib.plan_specs([s], 1, None, 1)
        o, k = db.offsets[t], s.numel
        so = db.scale_offsets[t]
        _, ns1 = oracle_lib.scale_offsets([s])
        _, nst1 = oracle_lib.state_offsets([s])
        hp_ = params[t].numpy().copy()
        mc = mc0[o:o + k].numpy().copy()
        vc = vc0[o:o + k].numpy().copy()
        ms = ms0[so:so + max(ns1, 1)].numpy().copy() if s.quant else np.zeros(1, np.float32)
        vs = vs0[so:so + max(ns1, 1)].numpy().copy() if s.quant else np.zeros(1, np.float32)
        m32 = np.zeros(max(nst1, 1), np.float32)
        v32 = np.zeros(max(nst1, 1), np.float32)
        oracle_lib.adamw8(sp, [s], hp_, grads[t].numpy().copy(), mc, vc, ms, vs, m32, v32,
                          lr=HP["lr"], beta1=b1, beta2=b2, eps=HP["eps"],
                          weight_decay=HP["weight_decay"], step=3, max_norm=0.5,
                          total_norm=0.75)
        assert_bits_equal(f32(p[o:o + k]), hp_, f"params t{t}")
        if s.quant:
            assert np.array_equal(st["m_codes"][o:o + k].cpu().numpy(), mc), f"m codes t{t}"
            assert np.array_equal(st["v_codes"][o:o + k].cpu().numpy(), vc), f"v codes t{t}"
            assert_bits_equal(f32(st["m_scales"][so:so + ns1]), ms[:ns1], f"m scales t{t}")
            assert_bits_equal(f32(st["v_scales"][so:so + ns1]), vs[:ns1], f"v scales t{t}")
        else:
            so32 = db.state_offsets[t]
            assert_bits_equal(f32(st["m32"][so32:so32 + k]), m32[:k], f"m32 t{t}")
            assert_bits_equal(f32(st["v32"][so32:so32 + k]), v32[:k], f"v32 t{t}")


def test_adamw8_every_group_size_in_one_launch(dbuf_lib, oracle_lib):
    """Blocks of 16 to 8192 elements in one plan: threads per block 1, 8, 16,
    32, 64, 128, 256 and 512 in the pipelined kernel, two-row blocks included,
    with more stages than SMs so that one CTA moves between tensors (and
    named-barrier ranges) from stage to stage; and the same plan through the
    register kernel (unaligned buffers)."""
    specs = [
        TensorSpec("s64x64", 768, 640, 64, qblock=(64, 64), quant="int8"),      # 256 threads/block
        TensorSpec("s64x128", 512, 1024, 64, qblock=(64, 128), quant="int8"),   # 512
        TensorSpec("s32x64", 640, 768, 32, qblock=(32, 64), quant="int8"),      # 128
        TensorSpec("vec", 1000, 1, 1),
        TensorSpec("s16x16", 400, 1280, 16, qblock=(16, 16), quant="int8"),     # 16
        TensorSpec("s32x32", 704, 704, 32, qblock=(32, 32), quant="int8"),      # 64
        TensorSpec("s1x16", 1024, 512, 1, qblock=(1, 16), quant="int8"),        # 1
        TensorSpec("s16x32", 336, 416, 16, qblock=(16, 32), quant="int8"),      # 32
        TensorSpec("s4x128", 36, 896, 4, qblock=(4, 128), quant="int8"),        # 32
        # two-row blocks whose rows hold more units than the block has threads: a
        # thread's units continue on the block's second row
        TensorSpec("s2x64", 258, 640, 2, qblock=(2, 64), quant="int8"),         # 8
        TensorSpec("s2x128", 130, 1152, 2, qblock=(2, 128), quant="int8"),      # 16
        TensorSpec("s4x32", 100, 160, 4, qblock=(4, 32), quant="int8"),         # 8
    ]
    c = Case(oracle_lib, specs, 4, seed=9)
    c.step(1, clip=True)
    c.step(2)
    c = Case(oracle_lib, specs, 3, seed=10, shift=1)
    c.step(1)


@pytest.mark.parametrize("hp,steps", [
    (dict(lr=3e-4, betas=(0.8, 0.999), eps=1e-6, weight_decay=0.0), (1, 2, 3)),
    (dict(lr=1e-2, betas=(0.95, 0.99), eps=0.0, weight_decay=0.5), (1, 7)),
    # late steps: both bias corrections near 1
    (dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1), (500, 5000)),
])
def test_adamw8_hyperparameters(dbuf_lib, oracle_lib, hp, steps):
    """Other betas, eps (0 included), weight decay and late steps, on block
    shapes of the pipelined kernel (its step scalars are computed on the host)
    and on those of the register kernel, against the oracle."""
    specs = [
        TensorSpec("s32x32", 160, 224, 32, qblock=(32, 32), quant="int8"),
        TensorSpec("s1x128", 40, 384, 1, qblock=(1, 128), quant="int8"),
        TensorSpec("vec", 300, 1, 1),
        TensorSpec("s128", 256, 136, 128, qblock=(128, 128), quant="int8"),
    ]
    c = Case(oracle_lib, specs, 4, seed=11)
    for i, st in enumerate(steps):
        c.step(st, clip=(i % 2 == 1), hp=hp)



def test_adamw8_more_tensors_than_one_launch_holds(dbuf_lib, oracle_lib):
    """41 quantised tensors of the pipelined kernel (three launches of at most 16
    tensors each, shapes and block shapes changing across the batch boundaries)
    with vectors between them, against the oracle; then the same plan through
    the register kernel (unaligned buffers)."""
    specs = []
    for i in range(41):
        qb = [(32, 32), (1, 128), (16, 64)][i % 3]
        rows = qb[0] * (2 + i % 5) + (7 if qb[0] == 1 else 0)
        specs.append(TensorSpec(f"w{i}", rows, 128 * (1 + i % 3), qb[0], qblock=qb, quant="int8"))
        if i % 7 == 3:
            specs.append(TensorSpec(f"b{i}", 96 + i, 1, 1))
    c = Case(oracle_lib, specs, 4, seed=12)
    c.step(1, clip=True)
    c.step(2)
    c = Case(oracle_lib, specs, 4, seed=13, shift=1)
    c.step(1)


# Blocks of 16384 elements (128x128, 64x256, 256x64) with 16-byte rows take the
# big-block pipelined kernel: gradients and codes staged whole, parameters read
# directly, two passes over one block per CTA at a time.
BIG = [
    TensorSpec("b128", 384, 256, 128, qblock=(128, 128), quant="int8"),
    TensorSpec("bias", 77, 1, 1),
    TensorSpec("b_edge", 300, 208, 128, qblock=(128, 128), quant="int8"),   # ragged edges
    TensorSpec("b64x256", 192, 512, 64, qblock=(64, 256), quant="int8"),
    TensorSpec("b256x64", 512, 128, 256, qblock=(256, 64), quant="int8"),
    TensorSpec("norm", 208, 1, 0, kind="norm"),
    TensorSpec("b_zero", 384, 128, 128, qblock=(128, 128), quant="int8"),
    TensorSpec("w_tiny", 256, 128, 128, qblock=(128, 128), quant="int8"),   # tiny values
    TensorSpec("w_sq", 96, 64, 32, qblock=(32, 32), quant="int8"),          # the stage kernel
]


def test_adamw8_big_blocks_steps(dbuf_lib, oracle_lib):
    c = Case(oracle_lib, BIG, 3, seed=21)
    assert len(c.db.specs) == len(BIG)
    for step, (clip, skip) in enumerate([(False, False), (True, False), (True, True),
                                         (False, False)], start=1):
        c.step(step, clip, skip)


def test_adamw8_big_blocks_zero_state_and_uneven_units(dbuf_lib, oracle_lib):
    c = Case(oracle_lib, BIG, 4, units=[2, 1, 3, 1], zero=True, seed=22)
    c.step(1, clip=True)
    c.step(2)


def test_adamw8_big_blocks_unaligned_take_the_register_kernel(dbuf_lib, oracle_lib):
    c = Case(oracle_lib, BIG, 3, seed=23, shift=1)
    c.step(1, clip=True)
    c.step(2)


def test_adamw8_big_blocks_two_launches(dbuf_lib, oracle_lib):
    """19 big-block tensors: two launches of at most 16 tensors' maps."""
    specs = []
    for i in range(19):
        qb = [(128, 128), (64, 256), (256, 64)][i % 3]
        specs.append(TensorSpec(f"w{i}", qb[0] * (1 + i % 3) + (40 if i % 4 == 1 else 0),
                                qb[1] * (1 + i % 2), qb[0], qblock=qb, quant="int8"))
        if i % 6 == 2:
            specs.append(TensorSpec(f"v{i}", 33 + i, 1, 1))
    c = Case(oracle_lib, specs, 4, seed=24)
    c.step(1)
    c.step(2, clip=True)


def test_adamw8_llama_layer_128x128(dbuf_lib, oracle_lib):
    g = adam8_group(workload("llama_layer").groups[0], (128, 128))
    c = Case(oracle_lib, list(g.tensors), 8, seed=25)
    c.step(3, clip=True)
