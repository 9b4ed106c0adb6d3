"""Pins of the oracle's fused AdamW step (no GPU).

- torch.optim.AdamW on the CPU (fp32, decoupled weight decay), a library routine:
  five steps agree to within rounding-order differences, so a wrong sign, a
  dropped term or a swapped beta would show.
- exact special cases: a skipped step (non-finite flag) writes nothing; lr = 0
  leaves parameters bitwise unchanged; with beta1 = beta2 = 0 the states are g
  and g*g; the first step moves each parameter by lr*sign(g) (|g| >> eps) plus
  decay; the clip coefficient matches torch.nn.utils.clip_grad_norm_; padding is
  untouched.
"""
import math

import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec


def _plan(oracle_lib, sizes, m=3, align=16):
    specs = [TensorSpec(f"t{i}", n, 1, 1) for i, n in enumerate(sizes)]
    return specs, oracle_lib.plan_specs(specs, m, None, align)


def _gather(p, a, specs):
    return np.concatenate([a[int(o):int(o) + s.numel] for o, s in zip(p.offsets, specs)])


def test_adamw_matches_torch(oracle_lib):
    rng = np.random.default_rng(0)
    sizes = [1000, 37, 4096]
    specs, p = _plan(oracle_lib, sizes)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    params = np.zeros(p.total, np.float32)
    m = np.zeros(p.total, np.float32)
    v = np.zeros(p.total, np.float32)
    for o, s in zip(p.offsets, specs):
        params[int(o):int(o) + s.numel] = rng.standard_normal(s.numel).astype(np.float32) * 0.02
    tparams = [torch.tensor(params[int(o):int(o) + s.numel]) for o, s in zip(p.offsets, specs)]
    for t in tparams:
        t.requires_grad_(True)
    opt = torch.optim.AdamW(tparams, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                            foreach=False)
    for step in range(1, 6):
        grad = np.zeros(p.total, np.float32)
        for (o, s), tp in zip(zip(p.offsets, specs), tparams):
            g = (rng.standard_normal(s.numel) * 1e-3).astype(np.float32)
            grad[int(o):int(o) + s.numel] = g
            tp.grad = torch.from_numpy(g.copy())
        opt.step()
        oracle_lib.adamw(p, params, grad, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps,
                         weight_decay=wd, step=step)
    got = _gather(p, params, specs)
    want = np.concatenate([t.detach().numpy() for t in tparams])
    # the update is lr-sized: differences of rounding order stay far below it
    assert np.max(np.abs(got - want)) <= 1e-3 * lr
    ms = np.concatenate([opt.state[t]["exp_avg"].numpy() for t in tparams])
    vs = np.concatenate([opt.state[t]["exp_avg_sq"].numpy() for t in tparams])
    # m and v are sums of gradient-sized terms (|g| ~ 1e-3) with cancellation in
    # m: compare at the rounding size of those terms; a wrong beta or a dropped
    # term would be off by ~1e-5 (m) and ~1e-8 (v)
    assert np.max(np.abs(_gather(p, m, specs) - ms)) <= 1e-9
    assert np.max(np.abs(_gather(p, v, specs) - vs)) <= 1e-12


def test_adamw_skip_zero_lr_and_padding(oracle_lib):
    rng = np.random.default_rng(1)
    specs, p = _plan(oracle_lib, [33, 64, 5])
    params = rng.standard_normal(p.total).astype(np.float32)
    grad = rng.standard_normal(p.total).astype(np.float32)
    m = rng.standard_normal(p.total).astype(np.float32)
    v = np.abs(rng.standard_normal(p.total)).astype(np.float32)
    ref = [a.copy() for a in (params, grad, m, v)]
    kw = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
    oracle_lib.adamw(p, params, grad, m, v, nonfinite=1, **kw)          # skipped step
    for a, r in zip((params, grad, m, v), ref):
        assert np.array_equal(a.view(np.uint32), r.view(np.uint32))
    kw["lr"] = 0.0
    oracle_lib.adamw(p, params, grad, m, v, **kw)                       # lr = 0
    assert np.array_equal(params.view(np.uint32), ref[0].view(np.uint32))
    # padding (outside every tensor range) is untouched in m and v too
    mask = np.ones(p.total, bool)
    for o, s in zip(p.offsets, specs):
        mask[int(o):int(o) + s.numel] = False
    assert mask.any()
    assert np.array_equal(m[mask], ref[2][mask]) and np.array_equal(v[mask], ref[3][mask])


def test_adamw_zero_betas_states_are_g_and_g_squared(oracle_lib):
    rng = np.random.default_rng(2)
    specs, p = _plan(oracle_lib, [500])
    o = int(p.offsets[0])
    params = np.zeros(p.total, np.float32)
    grad = np.zeros(p.total, np.float32)
    g = rng.standard_normal(500).astype(np.float32)
    grad[o:o + 500] = g
    m = np.full(p.total, 7.0, np.float32)
    v = np.full(p.total, 7.0, np.float32)
    oracle_lib.adamw(p, params, grad, m, v, lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8,
                     weight_decay=0.0, step=1)
    assert np.array_equal(m[o:o + 500], g)
    assert np.array_equal(v[o:o + 500], g * g)


def test_adamw_first_step_closed_form(oracle_lib):
    """Step 1 with bias correction: m_hat = g, v_hat = g^2, so the update is
    lr * g / (|g| + eps) = lr * sign(g) for |g| >> eps, on top of the decay."""
    rng = np.random.default_rng(3)
    specs, p = _plan(oracle_lib, [300])
    o = int(p.offsets[0])
    lr, wd = 1e-2, 0.1
    params = np.zeros(p.total, np.float32)
    p0 = rng.standard_normal(300).astype(np.float32)
    params[o:o + 300] = p0
    grad = np.zeros(p.total, np.float32)
    g = rng.choice([-1.0, 1.0], 300).astype(np.float32) * rng.uniform(0.5, 2.0, 300).astype(np.float32)
    grad[o:o + 300] = g
    m = np.zeros(p.total, np.float32)
    v = np.zeros(p.total, np.float32)
    b1, b2 = 0.9, 0.999
    oracle_lib.adamw(p, params, grad, m, v, lr=lr, beta1=b1, beta2=b2, eps=1e-8, weight_decay=wd,
                     step=1)
    want = p0.astype(np.float64) * (1 - lr * wd) - lr * np.sign(g)
    assert np.max(np.abs(params[o:o + 300] - want)) < 1e-6


@pytest.mark.parametrize("max_norm,total", [(1.0, 3.0), (1.0, 0.5), (0.0, 7.0), (2.5, 2.5)])
def test_clip_coef_matches_torch(oracle_lib, max_norm, total):
    c = oracle_lib.clip_coef(max_norm, total)
    if max_norm <= 0:
        assert c == 1.0
        return
    # torch.nn.utils.clip_grad_norm_ scales by min(1, max_norm / (norm + 1e-6))
    g = torch.zeros(1, dtype=torch.float32)
    g[0] = total
    g.requires_grad_(False)
    x = torch.nn.Parameter(torch.zeros(1))
    x.grad = g.clone()
    torch.nn.utils.clip_grad_norm_([x], max_norm)
    assert math.isclose(c * total, float(x.grad[0]), rel_tol=1e-6)
    assert c <= 1.0
