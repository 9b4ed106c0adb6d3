"""Rank-local operators on the GPU: every group operator run with a slice plan
(dbuf_plan_slice: shard k as a rank's local buffer) against the oracle's
whole-buffer result restricted to [B_k, B_{k+1}).

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer (each
rank owns one slice of the flat buffer), §4 and §6.3 (no block crosses a shard,
so each rank quantises its slice without communication).

Each local buffer sits between two guard regions filled with sentinels that must
survive; user tensors written by unpack keep their sentinel outside the slice's
piece.  Checked for every slice k of: the tiny two-layer group (E4M3 128x128,
m=4); an MoE-like group (row-wise units, uneven local_units, bf16 gradients,
INT8 1x128); a ragged group (odd vectors, E4M3 32x32 and INT8 4x16 blocks, an
empty and a whole tensor, m=5, alignment 4); the Llama layer (m=8); and seeded
random groups (eight by default, DBUF_RANDOM_CASES for more).  Per-piece
sums of squares added over the slices and finished by dbuf_norm_finish give
the whole group's norms (1e-5).  AdamW and 8-bit AdamW (32x32 INT8 blocks) run
on slices against the oracle's whole-buffer step.
"""
import os

import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import TensorSpec

from gpu_helpers import assert_norms_close, host_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
G = 256  # guard elements on each side of a local buffer


def _bits_fill(n, dtype, bits):
    if dtype == torch.bfloat16:
        return torch.full((n,), bits - (1 << 16) if bits >= 1 << 15 else bits, dtype=torch.int16,
                          device=DEV).view(torch.bfloat16)
    if dtype == torch.uint8:
        return torch.full((n,), bits, dtype=torch.uint8, device=DEV)
    return torch.full((n,), bits - (1 << 32) if bits >= 1 << 31 else bits, dtype=torch.int32,
                      device=DEV).view(torch.float32)


def _raw(x):
    x = x.detach().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).cpu().numpy().view(np.uint16)
    if x.dtype == torch.float32:
        return x.view(torch.int32).cpu().numpy().view(np.uint32)
    return x.cpu().numpy()


def _raw_np(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


class Guarded:
    """A local buffer of n elements between two guard regions of sentinels."""

    def __init__(self, n, dtype, bits, init=None):
        self.n, self.bits = n, bits
        self.big = _bits_fill(n + 2 * G, dtype, bits)
        self.buf = self.big[G:G + n]
        if init is not None:
            self.buf.copy_(init)

    def check(self, want_raw, what):
        got = _raw(self.big)
        sentinel = got[:1].copy()
        sentinel[0] = self.bits
        assert np.all(got[:G] == sentinel[0]) and np.all(got[G + self.n:] == sentinel[0]), \
            f"{what}: guard region written"
        bad = got[G:G + self.n] != want_raw
        assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, first at {np.nonzero(bad)[0][:6]}"


def _pieces(op, specs, k):
    B0, B1 = int(op.bounds[k]), int(op.bounds[k + 1])
    out = []
    for t, s in enumerate(specs):
        l = int(op.offsets[t])
        lo, hi = max(l, B0), min(l + s.numel, B1)
        out.append((lo - l, hi - lo, lo - B0) if hi > lo else (0, 0, 0))
    return B0, B1, out


def _oracle_slice_plan(oracle_lib, op, specs, k):
    B0, B1, pcs = _pieces(op, specs, k)
    return oracle_lib.Plan(B1 - B0, np.array([p[2] for p in pcs], np.int64),
                           np.array([0, B1 - B0], np.int64), np.array([p[1] for p in pcs], np.int64))


def _groups():
    tiny = workload("tiny")
    moe = [TensorSpec("router", 256, 8, 1, (1, 128), "int8")]
    for e in range(6):
        moe.append(TensorSpec(f"gate{e}", 256, 176, 1, (1, 128), "int8"))
        moe.append(TensorSpec(f"down{e}", 176, 256, 1, (1, 128), "int8"))
    ragged = [TensorSpec("v0", 1001, 1, 1), TensorSpec("q0", 96, 160, 32, (32, 32), "e4m3"),
              TensorSpec("v1", 7, 1, 1), TensorSpec("q1", 37, 48, 4, (4, 16), "int8"),
              TensorSpec("e", 0, 12, 1), TensorSpec("w", 13, 11, 0),
              TensorSpec("q2", 64, 100, 32, (32, 32), "e4m3"), TensorSpec("v2", 333, 1, 1)]
    ll = workload("llama_layer")
    return [("tiny", tiny.groups[0].tensors, tiny.m, None, tiny.align, torch.float32),
            ("moe_like", moe, 4, [1, 3, 2, 4], 16, torch.bfloat16),
            ("ragged", ragged, 5, None, 4, torch.float32),
            ("llama_layer", ll.groups[0].tensors, ll.m, None, ll.align, torch.float32)]


def _random_groups(n):
    """Seeded random groups of the kinds the random parity sweep draws (vectors,
    matrices at several row granularities, E4M3/INT8 blocks from 1x64 to
    128x128 and an odd 5x4, empty tensors, m 1..9, even or uneven units)."""
    from test_gpu_random import random_group
    out = []
    for i in range(n):
        rng = np.random.default_rng(3000 + i)
        specs, m, units, align = random_group(rng)
        gdt = torch.bfloat16 if rng.random() < 0.3 else torch.float32
        out.append((f"random{i}", specs, m, units, align, gdt))
    return out


# DBUF_RANDOM_CASES=N runs N random groups instead of the default 8
_NR = int(os.environ.get("DBUF_RANDOM_CASES", "0")) or 8


@pytest.mark.parametrize("case", range(4 + _NR))
def test_slice_operators_equal_the_whole_buffer(dbuf_lib, oracle_lib, case):
    from fsdp_infra_gb300 import DBuffer
    name, specs, m, units, align, gdt = (_groups() if case < 4 else _random_groups(case - 3))[
        case if case < 4 else -1]
    op = oracle_lib.plan_specs(specs, m, units, align)
    db = DBuffer(specs, m, units, align).upload()
    assert db.offsets == [int(x) for x in op.offsets]
    total = op.total
    gen = torch.Generator().manual_seed(50 + case)
    params = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    grads = [(torch.randn(s.rows, s.cols, generator=gen) * 1e-3).to(gdt) for s in specs]
    acc0 = torch.randn(total, generator=gen) * 1e-3

    # the oracle over the whole buffer (padding holds the same sentinels as the slices)
    w16 = np.full(total, 0xABCD, np.uint16)
    oracle_lib.pack(op, [p.reshape(-1).numpy() for p in params], w16)
    w32 = [np.full(s.numel, np.uint32(0x7FC0ABCD).view(np.float32), np.float32) for s in specs]
    oracle_lib.unpack(op, w16, w32)
    gbits = 0x7FC1 if gdt == torch.bfloat16 else 0x7FC0DEAD
    g_full = np.full(total, gbits, np.uint16 if gdt == torch.bfloat16 else np.uint32)
    a_full = np.full(total, 0x7FC0BEEF, np.uint32)
    for t, s in enumerate(specs):
        o = int(op.offsets[t])
        g_full[o:o + s.numel] = host_bits(grads[t]).reshape(-1).view(g_full.dtype)
        a_full[o:o + s.numel] = acc0[o:o + s.numel].numpy().view(np.uint32)
    g_in = g_full.copy()
    a_in = a_full.view(np.float32).copy()
    g_out, a_out = g_in.copy(), a_in.copy()
    g_host = g_out if gdt == torch.bfloat16 else g_out.view(np.float32)
    oracle_lib.scale_accum_zero(op, g_host, a_out, 1.0 / m)
    wn, wt, wf = oracle_lib.norm_nonfinite(op, a_out)
    assert wf == 0
    wcodes = np.full(total, 0x5A, np.uint8)
    wscales = oracle_lib.block_quant(op, specs, a_out, wcodes) if db.n_scales else None

    params_d = [p.to(DEV) for p in params]
    sumsq_all = torch.zeros(len(specs), dtype=torch.float64, device=DEV)
    scale_seen = 0
    for k in range(m):
        sl = db.slice(k).upload()
        B0, B1 = int(op.bounds[k]), int(op.bounds[k + 1])
        n = B1 - B0
        # pack fp32 -> bf16 into the local slice
        b = Guarded(n, torch.bfloat16, 0xABCD)
        sl.pack_cast(params_d, b.buf)
        torch.cuda.synchronize()
        b.check(w16[B0:B1], f"{name} pack k={k}")
        # unpack the slice into whole fp32 user tensors: only the piece is written
        dst = [_bits_fill(s.numel, torch.float32, 0x7FC0ABCD).view(s.rows, s.cols) for s in specs]
        sl.unpack(b.buf, dst)
        torch.cuda.synchronize()
        _, _, pcs = _pieces(op, specs, k)
        for t, (a, ln, _) in enumerate(pcs):
            want = np.full(specs[t].numel, 0x7FC0ABCD, np.uint32)
            want[a:a + ln] = w32[t].view(np.uint32)[a:a + ln]
            got = _raw(dst[t]).reshape(-1)
            assert np.array_equal(got, want), f"{name} unpack k={k} t={t}"
        # scale / accumulate / zero on the slice
        gl = Guarded(n, gdt, gbits, torch.from_numpy(g_in[B0:B1].view(
            np.int16 if gdt == torch.bfloat16 else np.int32)).to(DEV).view(gdt))
        al = Guarded(n, torch.float32, 0x7FC0BEEF, torch.from_numpy(a_in[B0:B1]).to(DEV))
        sl.scale_accum_zero(gl.buf, al.buf, 1.0 / m)
        torch.cuda.synchronize()
        gl.check(_raw_np(g_out[B0:B1]), f"{name} zero k={k}")
        al.check(a_out[B0:B1].view(np.uint32), f"{name} accumulate k={k}")
        # per-piece sums of squares (padding holds NaN: it must not be read)
        sumsq, flag = sl.norm_sumsq(al.buf)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0
        pn, _, pf = oracle_lib.norm_nonfinite(_oracle_slice_plan(oracle_lib, op, specs, k),
                                              a_out[B0:B1].copy())
        got = sumsq.cpu().numpy()
        want = np.asarray(pn, np.float64) ** 2
        assert np.all(np.abs(got - want) <= 2e-5 * want), f"{name} sumsq k={k}"
        sumsq_all += sumsq
        # block quantisation of the slice: local codes and a local range of scales
        if db.n_scales:
            cl = Guarded(n, torch.uint8, 0x5A)
            ns = sl.n_scales
            sc = Guarded(max(ns, 1), torch.float32, 0x7F80DEAD)
            sl.block_quant(al.buf, codes=cl.buf, scales=sc.buf)
            torch.cuda.synchronize()
            cl.check(wcodes[B0:B1], f"{name} codes k={k}")
            assert sl.scale_base == scale_seen
            if ns:
                sc.check(wscales[scale_seen:scale_seen + ns].view(np.uint32), f"{name} scales k={k}")
            scale_seen += ns
        sl.close()
    if db.n_scales:
        assert scale_seen == wscales.size
    norms, tot = db.norm_finish(sumsq_all)
    torch.cuda.synchronize()
    assert_norms_close(norms.cpu().numpy(), tot.item(), wn, wt, what=f"{name} sharded norms")
    db.close()


def test_slice_adamw_and_adamw8(dbuf_lib, oracle_lib):
    """AdamW and 8-bit AdamW (32x32 INT8 blocks at 32-row units, vectors in
    compact fp32 moments) on each slice equal the oracle's whole-buffer step."""
    from fsdp_infra_gb300 import DBuffer
    specs = [TensorSpec("a", 128, 96, 32, (32, 32), "int8"), TensorSpec("v", 300, 1, 1),
             TensorSpec("b", 96, 64, 32, (32, 32), "int8"), TensorSpec("u", 45, 1, 1),
             TensorSpec("c", 64, 128, 32, (32, 32), "int8")]
    m, align = 3, 16
    op = oracle_lib.plan_specs(specs, m, None, align)
    db = DBuffer(specs, m, None, align).upload()
    total = op.total
    gen = torch.Generator().manual_seed(8)
    p0 = (torch.randn(total, generator=gen) * 0.02).numpy()
    g0 = (torch.randn(total, generator=gen) * 1e-3).numpy()
    m0 = (torch.randn(total, generator=gen) * 1e-4).numpy()
    v0 = (torch.rand(total, generator=gen) * 1e-7).numpy()
    so, n_state = oracle_lib.state_offsets(specs)
    mc0 = torch.randint(0, 256, (total,), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
    vc0 = torch.randint(0, 256, (total,), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
    ms0 = (torch.rand(db.n_scales, generator=gen) * 1e-5 + 1e-7).numpy()
    vs0 = (torch.rand(db.n_scales, generator=gen) * 1e-9 + 1e-12).numpy()
    m320 = (torch.randn(max(n_state, 1), generator=gen) * 1e-4).numpy()
    v320 = (torch.rand(max(n_state, 1), generator=gen) * 1e-7).numpy()
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=3)
    # the whole-buffer oracle steps
    pa, ma, va = p0.copy(), m0.copy(), v0.copy()
    oracle_lib.adamw(op, pa, g0.copy(), ma, va, **hp)
    p8, mc, vc, ms, vs, m32, v32 = (p0.copy(), mc0.copy(), vc0.copy(), ms0.copy(), vs0.copy(),
                                    m320.copy(), v320.copy())
    oracle_lib.adamw8(op, specs, p8, g0.copy(), mc, vc, ms, vs, m32, v32, **hp)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    step_kw = dict(step=hp["step"], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                   weight_decay=hp["weight_decay"])
    for k in range(m):
        sl = db.slice(k).upload()
        B0, B1 = int(op.bounds[k]), int(op.bounds[k + 1])
        # fp32 AdamW
        p, g, mm, vv = dev(p0[B0:B1]), dev(g0[B0:B1]), dev(m0[B0:B1]), dev(v0[B0:B1])
        sl.adamw_step(p, g, mm, vv, **step_kw)
        torch.cuda.synchronize()
        for x, w, nm in ((p, pa, "p"), (mm, ma, "m"), (vv, va, "v")):
            assert np.array_equal(_raw(x), w[B0:B1].view(np.uint32)), f"adamw {nm} k={k}"
        # 8-bit AdamW: the slice's state is the whole state's slice (compact fp32
        # moments re-indexed by the slice's own compact layout)
        _, _, pcs = _pieces(op, specs, k)
        lm32 = np.zeros(max(sl.n_state, 1), np.float32)
        lv32 = np.zeros(max(sl.n_state, 1), np.float32)
        for t, (a, ln, _) in enumerate(pcs):
            if not specs[t].quant and ln:
                ls = sl.state_offsets[t]
                lm32[ls:ls + ln] = m320[so[t] + a:so[t] + a + ln]
                lv32[ls:ls + ln] = v320[so[t] + a:so[t] + a + ln]
        sb, ns = sl.scale_base, sl.n_scales
        st = {"m_codes": dev(mc0[B0:B1]), "v_codes": dev(vc0[B0:B1]),
              "m_scales": dev(ms0[sb:sb + ns]), "v_scales": dev(vs0[sb:sb + ns]),
              "m32": dev(lm32), "v32": dev(lv32)}
        p = dev(p0[B0:B1])
        sl.adamw8_step(p, dev(g0[B0:B1]), st, **step_kw)
        torch.cuda.synchronize()
        assert np.array_equal(_raw(p), p8[B0:B1].view(np.uint32)), f"adamw8 p k={k}"
        assert np.array_equal(st["m_codes"].cpu().numpy(), mc[B0:B1]), f"adamw8 m codes k={k}"
        assert np.array_equal(st["v_codes"].cpu().numpy(), vc[B0:B1]), f"adamw8 v codes k={k}"
        assert np.array_equal(_raw(st["m_scales"]), ms[sb:sb + ns].view(np.uint32))
        assert np.array_equal(_raw(st["v_scales"]), vs[sb:sb + ns].view(np.uint32))
        got_m, got_v = st["m32"].cpu().numpy(), st["v32"].cpu().numpy()
        for t, (a, ln, _) in enumerate(pcs):
            if not specs[t].quant and ln:
                ls = sl.state_offsets[t]
                assert np.array_equal(got_m[ls:ls + ln].view(np.uint32),
                                      m32[so[t] + a:so[t] + a + ln].view(np.uint32))
                assert np.array_equal(got_v[ls:ls + ln].view(np.uint32),
                                      v32[so[t] + a:so[t] + a + ln].view(np.uint32))
        sl.close()
    db.close()
