"""Pins of the oracle's 8-bit AdamW step (no GPU).

- the second moment's code map against brute force: the code is the nearest of
  the 256 levels (c + 1) * scale to v (ties to the even level), never a level
  below the first, and 0 for an all-zero block;
- the step is the composition of independently pinned pieces: dequantise with
  numpy, the fp32 AdamW step (pinned against torch.optim.AdamW), re-encode m with
  the INT8 block quantiser (pinned against numpy's rint) and v with the code map
  above; parameters, codes, scales and the compact fp32 states must agree bit
  for bit, on ragged edge blocks, row blocks and square blocks;
- closed forms of the first step from a zero state: dequantised moments within
  half a level of (1 - beta1) g and (1 - beta2) g^2, no positive v at zero, the
  block maximum at code 127 / 255;
- a skipped step writes nothing; bytes outside quantised tensors are untouched;
- over 30 steps on Gaussian gradients the 8-bit trajectory stays close to the
  fp32 one (the reason the second moment's map has no zero level).
"""
import numpy as np
import pytest

from workloads.configs import TensorSpec

HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _specs():
    return [
        TensorSpec("w_sq", 70, 96, 32, qblock=(32, 32), quant="int8"),       # ragged last block row
        TensorSpec("bias", 57, 1, 1),
        TensorSpec("w_row", 33, 130, 1, qblock=(1, 128), quant="e4m3"),      # 2-column edge blocks
        TensorSpec("empty", 0, 64, 32, qblock=(32, 32), quant="int8"),
        TensorSpec("w_odd", 15, 7, 5, qblock=(5, 3), quant="int8"),          # odd block widths
        TensorSpec("norm", 96, 1, 0, kind="norm"),
        TensorSpec("w_full", 8, 40, 8, qblock=(8, 0), quant="int8"),         # block = 8 full rows
    ]


def _blocks(s):
    qr = s.qblock[0] if s.qblock[0] > 0 else s.rows
    qc = s.qblock[1] if s.qblock[1] > 0 else s.cols
    for r0 in range(0, s.rows, max(qr, 1)):
        for c0 in range(0, s.cols, max(qc, 1)):
            yield slice(r0, min(r0 + qr, s.rows)), slice(c0, min(c0 + qc, s.cols))


def _state(oracle_lib, specs, p, rng, zero=False):
    so, n_state = oracle_lib.state_offsets(specs)
    _, n_scales = oracle_lib.scale_offsets(specs)
    st = {
        "p": np.zeros(p.total, np.float32), "mc": np.zeros(p.total, np.uint8),
        "vc": np.zeros(p.total, np.uint8), "ms": np.zeros(max(n_scales, 1), np.float32),
        "vs": np.zeros(max(n_scales, 1), np.float32), "m32": np.zeros(max(n_state, 1), np.float32),
        "v32": np.zeros(max(n_state, 1), np.float32),
    }
    for o, s in zip(p.offsets, specs):
        st["p"][int(o):int(o) + s.numel] = rng.standard_normal(s.numel).astype(np.float32) * 0.02
    if not zero:
        for o, s in zip(p.offsets, specs):
            if s.quant is None:
                continue
            st["mc"][int(o):int(o) + s.numel] = rng.integers(-127, 128, s.numel).astype(np.int8).view(np.uint8)
            st["vc"][int(o):int(o) + s.numel] = rng.integers(0, 256, s.numel).astype(np.uint8)
        st["ms"][:n_scales] = rng.uniform(1e-7, 1e-5, n_scales).astype(np.float32)
        st["vs"][:n_scales] = rng.uniform(1e-12, 1e-9, n_scales).astype(np.float32)
        st["m32"][:] = rng.standard_normal(st["m32"].size).astype(np.float32) * 1e-4
        st["v32"][:] = np.abs(rng.standard_normal(st["v32"].size)).astype(np.float32) * 1e-8
    return st


def _grad(p, specs, rng, std=1e-3):
    g = np.zeros(p.total, np.float32)
    for o, s in zip(p.offsets, specs):
        g[int(o):int(o) + s.numel] = (rng.standard_normal(s.numel) * std).astype(np.float32)
    return g


def _step8(oracle_lib, p, specs, st, g, step, **kw):
    b1, b2 = HP["beta1"], HP["beta2"]
    oracle_lib.adamw8(p, specs, st["p"], g, st["mc"], st["vc"], st["ms"], st["vs"], st["m32"],
                      st["v32"], **HP, step=step, **kw)


def test_v_code_is_the_nearest_nonzero_level(oracle_lib):
    rng = np.random.default_rng(0)
    levels = np.arange(1, 257, dtype=np.float64)
    for scale in [np.float32(3e-9), np.float32(0.37), np.float32(1.0), np.float32(2.0 ** -100)]:
        amax = np.float32(scale * 256)
        vs = np.concatenate([rng.uniform(0, float(amax), 300),
                             np.float32(scale) * (np.arange(0, 258) + 0.5),     # ties
                             [0.0, float(amax), float(scale) * 1e-3]]).astype(np.float32)
        for v in vs:
            q = float(np.float32(v) / np.float32(scale))                      # the fp32 quotient
            d = np.abs(levels - q)
            best = np.flatnonzero(d == d.min())
            c = int(best[0]) if len(best) == 1 else int(best[levels[best] % 2 == 0][0])
            assert oracle_lib.v_code(float(v), float(scale)) == c, (scale, v)
    assert oracle_lib.v_code(0.0, 0.0) == 0
    assert oracle_lib.v_code(1e-30, 1.0) == 0            # below the first level: level 1
    assert oracle_lib.v_code(1e9, 1.0) == 255            # above the last: clamped


def test_state_offsets_layout(oracle_lib):
    specs = _specs()
    so, total = oracle_lib.state_offsets(specs)
    end = 0
    for s, o in zip(specs, so):
        if s.quant is not None:
            assert o == -1
            continue
        assert o % 4 == 0 and o >= end
        end = o + s.numel
    assert total == (end + 3) // 4 * 4


def test_adamw8_is_dequantise_adamw_requantise(oracle_lib):
    rng = np.random.default_rng(1)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, 3, None, 16)
    so, _ = oracle_lib.state_offsets(specs)
    soff, _ = oracle_lib.scale_offsets(specs)
    st = _state(oracle_lib, specs, p, rng)
    g = _grad(p, specs, rng)
    # expected: dequantise (numpy fp32), fp32 AdamW step, re-encode
    m = np.zeros(p.total, np.float32)
    v = np.zeros(p.total, np.float32)
    for t, (o, s) in enumerate(zip(p.offsets, specs)):
        o = int(o)
        if s.quant is None:
            m[o:o + s.numel] = st["m32"][so[t]:so[t] + s.numel]
            v[o:o + s.numel] = st["v32"][so[t]:so[t] + s.numel]
            continue
        mc = st["mc"][o:o + s.numel].view(np.int8).astype(np.float32).reshape(s.rows, s.cols)
        vc = st["vc"][o:o + s.numel].astype(np.float32).reshape(s.rows, s.cols)
        mm = np.zeros_like(mc)
        vv = np.zeros_like(vc)
        for b, (rs, cs) in enumerate(_blocks(s)):
            mm[rs, cs] = mc[rs, cs] * st["ms"][soff[t] + b]
            vv[rs, cs] = (vc[rs, cs] + np.float32(1)) * st["vs"][soff[t] + b]
        m[o:o + s.numel] = mm.reshape(-1)
        v[o:o + s.numel] = vv.reshape(-1)
    pw = st["p"].copy()
    oracle_lib.adamw(p, pw, g, m, v, **HP, step=4, max_norm=0.05, total_norm=0.2)
    int8_specs = [TensorSpec(s.name, s.rows, s.cols, s.gran_rows, s.qblock, "int8" if s.quant else None)
                  for s in specs]
    want_mc = np.zeros(p.total, np.uint8)
    want_ms = oracle_lib.block_quant(p, int8_specs, m, want_mc)
    _step8(oracle_lib, p, specs, st, g, 4, max_norm=0.05, total_norm=0.2)
    for t, (o, s) in enumerate(zip(p.offsets, specs)):
        o = int(o)
        sl = slice(o, o + s.numel)
        assert np.array_equal(st["p"][sl].view(np.uint32), pw[sl].view(np.uint32)), s.name
        if s.quant is None:
            assert np.array_equal(st["m32"][so[t]:so[t] + s.numel], m[sl]), s.name
            assert np.array_equal(st["v32"][so[t]:so[t] + s.numel], v[sl]), s.name
            continue
        assert np.array_equal(st["mc"][sl], want_mc[sl]), s.name
        vv = v[sl].reshape(s.rows, s.cols)
        vc = st["vc"][sl].reshape(s.rows, s.cols)
        for b, (rs, cs) in enumerate(_blocks(s)):
            k = soff[t] + b
            assert st["ms"][k] == want_ms[k]
            scale = np.float32(np.max(vv[rs, cs]) / np.float32(256))
            assert st["vs"][k] == scale
            want = [oracle_lib.v_code(float(x), float(scale)) for x in vv[rs, cs].reshape(-1)]
            assert np.array_equal(vc[rs, cs].reshape(-1), np.array(want, np.uint8)), (s.name, b)


def test_adamw8_first_step_closed_form(oracle_lib):
    rng = np.random.default_rng(2)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, 2, None, 16)
    soff, _ = oracle_lib.scale_offsets(specs)
    st = _state(oracle_lib, specs, p, rng, zero=True)
    g = _grad(p, specs, rng)
    # zero codes with zero scales dequantise to exact zeros: the parameters move
    # exactly as the fp32 step from zero moments
    pw = st["p"].copy()
    oracle_lib.adamw(p, pw, g, np.zeros(p.total, np.float32), np.zeros(p.total, np.float32), **HP,
                     step=1)
    _step8(oracle_lib, p, specs, st, g, 1)
    for t, (o, s) in enumerate(zip(p.offsets, specs)):
        sl = slice(int(o), int(o) + s.numel)
        assert np.array_equal(st["p"][sl].view(np.uint32), pw[sl].view(np.uint32)), s.name
        if s.quant is None or s.numel == 0:
            continue
        gg = g[sl].astype(np.float64).reshape(s.rows, s.cols)
        mc = st["mc"][sl].view(np.int8).reshape(s.rows, s.cols).astype(np.float64)
        vc = st["vc"][sl].reshape(s.rows, s.cols).astype(np.float64)
        for b, (rs, cs) in enumerate(_blocks(s)):
            ms, vs = float(st["ms"][soff[t] + b]), float(st["vs"][soff[t] + b])
            m1 = 0.1 * gg[rs, cs]
            v1 = 0.05 * gg[rs, cs] ** 2
            assert np.max(np.abs(mc[rs, cs] * ms - m1)) <= 0.5 * ms * (1 + 1e-5)
            assert np.max(np.abs(np.maximum(vc[rs, cs] + 1, 1) * vs - v1)) <= 0.5 * vs * (1 + 1e-5) + \
                np.max(np.where(v1 < vs, vs - v1, 0))
            assert np.max(np.abs(mc[rs, cs])) == 127 and np.max(vc[rs, cs]) == 255
            assert np.all((vc[rs, cs] + 1) * vs > 0)


def test_adamw8_skip_and_untouched_bytes(oracle_lib):
    rng = np.random.default_rng(3)
    specs = _specs()
    p = oracle_lib.plan_specs(specs, 3, None, 16)
    st = _state(oracle_lib, specs, p, rng)
    # fill the bytes outside quantised tensors with a marker
    outside = np.ones(p.total, bool)
    for o, s in zip(p.offsets, specs):
        if s.quant is not None:
            outside[int(o):int(o) + s.numel] = False
    st["mc"][outside] = 0xA5
    st["vc"][outside] = 0x5A
    ref = {k: a.copy() for k, a in st.items()}
    g = _grad(p, specs, rng)
    _step8(oracle_lib, p, specs, st, g, 2, nonfinite=1)
    for k in st:
        assert np.array_equal(st[k].view(np.uint8), ref[k].view(np.uint8)), k
    _step8(oracle_lib, p, specs, st, g, 2)
    assert np.all(st["mc"][outside] == 0xA5) and np.all(st["vc"][outside] == 0x5A)
    assert not np.array_equal(st["p"], ref["p"])


def test_adamw8_tracks_the_fp32_step(oracle_lib):
    """30 steps on Gaussian gradients of a 32x32-block tensor: the 8-bit
    trajectory stays within a small fraction of the distance the fp32 one
    travels (a second-moment level at zero would instead blow small-v elements
    up to steps of about lr * |m| / eps)."""
    rng = np.random.default_rng(4)
    specs = [TensorSpec("w", 128, 256, 32, qblock=(32, 32), quant="int8")]
    p = oracle_lib.plan_specs(specs, 2, None, 16)
    st = _state(oracle_lib, specs, p, rng, zero=True)
    p32 = st["p"].copy()
    p0 = p32.copy()
    m = np.zeros(p.total, np.float32)
    v = np.zeros(p.total, np.float32)
    for step in range(1, 31):
        g = _grad(p, specs, rng)
        _step8(oracle_lib, p, specs, st, g, step)
        oracle_lib.adamw(p, p32, g, m, v, **HP, step=step)
    travel = np.abs(p32 - p0)
    dev = np.abs(st["p"] - p32)
    assert np.max(dev) <= 0.5 * 30 * HP["lr"]
    assert np.mean(dev) <= 0.1 * np.mean(travel)
