"""GPU parity of the fused AdamW step (dbuf_adamw_step) against the oracle.

Bit-exact when both sides get the same clip norm (an fp32 value written from the
host, derived from the oracle's norm); within a tolerance set by the norm's
1e-5 relative bound when the kernel reads the GPU's own norm of the same
gradients, which is how the step is wired in training (no host round trip).
"""
import math

import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import TensorSpec, grad_values, param_values

from gpu_helpers import assert_bits_equal, f32

pytestmark = pytest.mark.gpu

DEV = "cuda"
HP = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)


def _db(specs, m, units=None, align=16):
    from fsdp_infra_gb300 import DBuffer
    return DBuffer(specs, m, units, align).upload()


def _fill(db, specs, values):
    buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    for t, x in enumerate(values):
        buf[db.offsets[t]:db.offsets[t] + specs[t].numel].copy_(x.reshape(-1).to(DEV))
    return buf


def _oracle_step(oracle_lib, op, host, step, max_norm=0.0, total=0.0, flag=0):
    b1, b2 = HP["betas"]
    oracle_lib.adamw(op, host["p"], host["g"], host["m"], host["v"], lr=HP["lr"], beta1=b1,
                     beta2=b2, eps=HP["eps"], weight_decay=HP["weight_decay"],
                     step=step, max_norm=max_norm, total_norm=total, nonfinite=flag)


def _run_steps(oracle_lib, specs, m, steps, units=None, align=16, shift=0):
    op = oracle_lib.plan_specs(specs, m, units, align)
    db = _db(specs, m, units, align)
    gen = torch.Generator().manual_seed(41)
    p = _fill(db, specs, [torch.randn(s.numel, generator=gen) * 0.02 for s in specs])
    mstate = torch.zeros(db.total + 8, dtype=torch.float32, device=DEV)[shift:shift + db.total]
    vstate = torch.zeros(db.total + 8, dtype=torch.float32, device=DEV)[shift:shift + db.total]
    host = {"p": f32(p).copy(), "m": f32(mstate).copy(), "v": f32(vstate).copy()}
    norm_dev = torch.zeros(1, dtype=torch.float32, device=DEV)
    flag_dev = torch.zeros(1, dtype=torch.int32, device=DEV)
    for step, (clip, skip) in enumerate(steps, start=1):
        g = _fill(db, specs, [torch.randn(s.numel, generator=gen) * 1e-3 for s in specs])
        host["g"] = f32(g).copy()
        wn, wt, _ = oracle_lib.norm_nonfinite(op, host["g"])
        total32 = float(np.float32(wt))
        norm_dev.fill_(total32)
        flag_dev.fill_(1 if skip else 0)
        max_norm = 0.5 * total32 if clip else 0.0
        db.adamw_step(p, g, mstate, vstate, step=step, max_norm=max_norm, total_norm=norm_dev,
                      nonfinite=flag_dev, **HP)
        _oracle_step(oracle_lib, op, host, step, max_norm, total32, 1 if skip else 0)
        assert_bits_equal(f32(p), host["p"], f"params step {step}")
        assert_bits_equal(f32(mstate), host["m"], f"exp_avg step {step}")
        assert_bits_equal(f32(vstate), host["v"], f"exp_avg_sq step {step}")
    return db


def test_adamw_tiny_group_steps(dbuf_lib, oracle_lib):
    w = workload("tiny")
    _run_steps(oracle_lib, w.groups[0].tensors, w.m,
               [(False, False), (True, False), (True, True), (False, False)])


def test_adamw_llama_layer_steps(dbuf_lib, oracle_lib):
    w = workload("llama_layer")
    _run_steps(oracle_lib, w.groups[0].tensors, w.m, [(True, False), (False, False), (True, False)])


def test_adamw_ragged_and_unaligned(dbuf_lib, oracle_lib):
    specs = [TensorSpec("a", 37, 3, 1), TensorSpec("b", 16384 + 5, 1, 1), TensorSpec("e", 0, 4, 1),
             TensorSpec("c", 130, 7, 0)]
    for m, align, shift in [(3, 16, 0), (5, 1, 0), (2, 16, 1)]:
        _run_steps(oracle_lib, specs, m, [(True, False), (False, False)], None, align, shift)


def test_adamw_wired_to_the_gpu_norm(dbuf_lib, oracle_lib):
    """Training wiring: the step reads the GPU's own norm and flag of the same
    gradients.  The norm is within 1e-5 relative of the oracle's, so the clipped
    update differs from the oracle's by at most that relative amount of lr."""
    w = workload("tiny")
    specs = w.groups[0].tensors
    op = oracle_lib.plan_specs(specs, w.m, None, w.align)
    db = _db(specs, w.m)
    p = _fill(db, specs, [param_values(w, 0, t) for t in range(len(specs))])
    g = _fill(db, specs, [grad_values(w, 0, t) for t in range(len(specs))])
    ms = torch.zeros_like(p)
    vs = torch.zeros_like(p)
    host = {"p": f32(p).copy(), "g": f32(g).copy(), "m": f32(ms).copy(), "v": f32(vs).copy()}
    norms, total, flag = db.norm_nonfinite(g)
    _, wt, wf = oracle_lib.norm_nonfinite(op, host["g"])
    max_norm = 0.25 * wt
    db.adamw_step(p, g, ms, vs, step=1, max_norm=max_norm, total_norm=total, nonfinite=flag, **HP)
    _oracle_step(oracle_lib, op, host, 1, max_norm, float(np.float32(wt)), wf)
    err = np.max(np.abs(f32(p) - host["p"]))
    assert err <= 1e-4 * HP["lr"]
    # an inf in the gradients raises the flag and the step writes nothing
    g[db.offsets[2] + 5] = float("inf")
    p0 = p.clone()
    norms, total, flag = db.norm_nonfinite(g)
    db.adamw_step(p, g, ms, vs, step=2, max_norm=max_norm, total_norm=total, nonfinite=flag, **HP)
    assert int(flag.item()) == 1 and torch.equal(p, p0)


def test_adamw_dense7b_layer_full_size(dbuf_lib, oracle_lib, oracle_plans):
    """One step on a full-size 7B-shaped layer DBuffer; each tensor checked
    against the oracle run on that tensor alone."""
    w = workload("dense7b")
    specs = w.groups[0].tensors
    op = oracle_plans("dense7b", 0)
    db = _db(specs, w.m)
    assert db.offsets == [int(x) for x in op.offsets]
    params = [param_values(w, 0, t, device=DEV).reshape(-1) for t in range(len(specs))]
    grads = [grad_values(w, 0, t, device=DEV).reshape(-1) for t in range(len(specs))]
    p = _fill(db, specs, params)
    g = _fill(db, specs, grads)
    ms = _fill(db, specs, [x * 0.5 for x in grads])
    vs = _fill(db, specs, [x * x for x in grads])
    total = torch.tensor([0.75], device=DEV)
    db.adamw_step(p, g, ms, vs, step=3, max_norm=0.5, total_norm=total, **HP)
    torch.cuda.synchronize()
    for t, s in enumerate(specs):
        sp = oracle_lib.plan_specs([s], 1, None, 1)
        o, k = db.offsets[t], s.numel
        host = {"p": f32(params[t]).copy(), "g": f32(grads[t]).copy(),
                "m": f32(grads[t] * 0.5).copy(), "v": f32(grads[t] * grads[t]).copy()}
        _oracle_step(oracle_lib, sp, host, 3, 0.5, 0.75)
        assert_bits_equal(f32(p[o:o + k]), host["p"], f"params t{t}")
        assert_bits_equal(f32(ms[o:o + k]), host["m"], f"exp_avg t{t}")
        assert_bits_equal(f32(vs[o:o + k]), host["v"], f"exp_avg_sq t{t}")
