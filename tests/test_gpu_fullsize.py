"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: the 7B-shaped dense layer and embedding DBuffers (m=64), the
MoE group (uneven local_units, bf16 grads, INT8 1x128) and the 2000-tensor mixed
group (m=32).  The layouts are compared whole.  The MoE and mixed groups run the
oracle once on the whole planned group and compare every operator's output over
the whole buffer, padding included: padding holds sentinels (NaN in the gradient
and accumulator) that must come back unchanged and must not raise the
non-finite flag.  The dense groups compare every tensor against the oracle run
on that tensor alone.  Norms and the non-finite flag are checked for every
tensor.  Inputs are drawn on the device by torch's seeded generator and copied
to the host for the oracle.
"""
import math

import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import param_values, grad_values

from gpu_helpers import assert_bits_equal, assert_norms_close, bf16_bits, f32, host_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _db(specs, m, units, align):
    from fsdp_infra_gb300 import DBuffer
    return DBuffer(specs, m, units, align).upload()


def _acc_values(w, gi, t, spec):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(777_000 + 1000 * gi + t)
    return torch.randn(spec.numel, generator=gen, device=DEV) * 1e-3


def sampled_group_parity(oracle_lib, op, w, gi, sample):
    g = w.groups[gi]
    specs = g.tensors
    n = len(specs)
    db = _db(specs, w.m, w.local_units, w.align)
    assert db.S == op.S and db.total == op.total
    assert db.offsets == [int(x) for x in op.offsets]
    assert db.shard_bounds == [int(x) for x in op.bounds]
    total = db.total

    params = [param_values(w, gi, t, device=DEV) for t in range(n)]
    buf16 = torch.zeros(total, dtype=torch.bfloat16, device=DEV)
    db.pack_cast(params, buf16)
    dst = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=DEV) for s in specs]
    db.unpack(buf16, dst)

    grads = [grad_values(w, gi, t, device=DEV) for t in range(n)]
    grad = torch.zeros(total, dtype=w.grad_dtype, device=DEV)
    acc = torch.zeros(total, dtype=torch.float32, device=DEV)
    accs = [_acc_values(w, gi, t, specs[t]) for t in sample]
    for t in range(n):
        grad[db.offsets[t]:db.offsets[t] + specs[t].numel].copy_(grads[t].reshape(-1))
    for t, a in zip(sample, accs):
        acc[db.offsets[t]:db.offsets[t] + specs[t].numel].copy_(a)

    norms, tot, flag = db.norm_nonfinite(grad)
    db.scale_accum_zero(grad, acc, w.scale)
    codes, scales = db.block_quant(acc) if db.n_scales else (None, None)
    torch.cuda.synchronize()

    # norms of every tensor: oracle on each tensor's generated gradient alone
    want_norms = np.zeros(n)
    for t in range(n):
        sp = oracle_lib.plan_specs([specs[t]], 1, None, 1)
        nn, _, wf = oracle_lib.norm_nonfinite(sp, host_bits(grads[t]).reshape(-1))
        assert wf == 0
        want_norms[t] = nn[0]
    assert int(flag.item()) == 0
    assert_norms_close(f32(norms), tot.item(), want_norms,
                       math.sqrt(float(np.sum(want_norms ** 2))), what=f"{w.key} norms")

    q_offsets, _ = oracle_lib.scale_offsets(specs)
    for t, a in zip(sample, accs):
        s = specs[t]
        sp = oracle_lib.plan_specs([s], 1, None, 1)
        o, k = db.offsets[t], s.numel
        # pack (fp32 -> bf16) and unpack (bf16 -> bf16)
        want16 = np.zeros(k, np.uint16)
        oracle_lib.pack(sp, [f32(params[t]).reshape(-1)], want16)
        assert_bits_equal(bf16_bits(buf16[o:o + k]), want16, f"{w.key} pack t{t}")
        wd = np.zeros(k, np.uint16)
        oracle_lib.unpack(sp, want16, [wd])
        assert_bits_equal(bf16_bits(dst[t]).reshape(-1), wd, f"{w.key} unpack t{t}")
        # scale / accumulate / zero
        g_h = host_bits(grads[t]).reshape(-1).copy()
        a_h = f32(a).copy()
        oracle_lib.scale_accum_zero(sp, g_h, a_h, w.scale)
        assert_bits_equal(f32(acc[o:o + k]), a_h, f"{w.key} accumulate t{t}")
        assert_bits_equal(host_bits(grad[o:o + k]), g_h, f"{w.key} zero t{t}")
        # block quantisation of the accumulator
        if s.quant:
            wc = np.zeros(k, np.uint8)
            ws = oracle_lib.block_quant(sp, [s], a_h, wc)
            so = int(q_offsets[t])
            assert_bits_equal(f32(scales[so:so + ws.size]), ws, f"{w.key} scales t{t}")
            assert_bits_equal(codes[o:o + k].cpu().numpy(), wc, f"{w.key} codes t{t}")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0
    del grad, acc, buf16, dst, codes
    torch.cuda.empty_cache()


def _fill_bits(n, dtype, bits):
    """A device buffer of n elements whose every element has the bit pattern `bits`."""
    if dtype == torch.bfloat16:
        return torch.full((n,), bits - (1 << 16) if bits >= 1 << 15 else bits, dtype=torch.int16,
                          device=DEV).view(torch.bfloat16)
    return torch.full((n,), bits - (1 << 32) if bits >= 1 << 31 else bits, dtype=torch.int32,
                      device=DEV).view(torch.float32)


def _raw(x: torch.Tensor) -> np.ndarray:
    """Host copy of a device buffer as raw unsigned bits."""
    x = x.detach().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).cpu().numpy().view(np.uint16)
    if x.dtype == torch.float32:
        return x.view(torch.int32).cpu().numpy().view(np.uint32)
    return x.cpu().numpy()


def _assert_raw_equal(got: np.ndarray, want: np.ndarray, what: str):
    bad = got != want
    if bad.any():
        idx = np.nonzero(bad)[0][:8]
        raise AssertionError(f"{what}: {int(bad.sum())} mismatches, first at {idx.tolist()}: "
                             f"got {[hex(int(v)) for v in got[idx]]} want {[hex(int(v)) for v in want[idx]]}")


def whole_group_parity(oracle_lib, op, w, gi):
    """Every operator of the step on the whole planned group, against the oracle
    run once on the whole group, compared over whole buffers (padding included)."""
    g = w.groups[gi]
    specs = g.tensors
    n = len(specs)
    db = _db(specs, w.m, w.local_units, w.align)
    assert db.S == op.S and db.total == op.total
    assert db.offsets == [int(x) for x in op.offsets]
    assert db.shard_bounds == [int(x) for x in op.bounds]
    total = db.total

    # pack fp32 -> bf16 into a buffer whose padding holds a sentinel, then unpack
    params = [param_values(w, gi, t, device=DEV) for t in range(n)]
    buf16 = _fill_bits(total, torch.bfloat16, 0xABCD)
    db.pack_cast(params, buf16)
    dst = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=DEV) for s in specs]
    db.unpack(buf16, dst)
    torch.cuda.synchronize()
    host_params = [f32(x).reshape(-1) for x in params]
    del params
    want16 = np.full(total, 0xABCD, np.uint16)
    oracle_lib.pack(op, host_params, want16)
    del host_params
    _assert_raw_equal(_raw(buf16), want16, f"{w.key} pack (whole buffer)")
    del buf16
    wd = [np.zeros(s.numel, np.uint16) for s in specs]
    oracle_lib.unpack(op, want16, wd)
    del want16
    _assert_raw_equal(np.concatenate([_raw(x).reshape(-1) for x in dst] or [np.zeros(0, np.uint16)]),
                      np.concatenate(wd or [np.zeros(0, np.uint16)]), f"{w.key} unpack (every tensor)")
    del dst, wd
    torch.cuda.empty_cache()

    # gradient and accumulator: NaN sentinels in the padding
    gbits = 0x7FC1 if w.grad_dtype == torch.bfloat16 else 0x7FC0DEAD
    grad = _fill_bits(total, w.grad_dtype, gbits)
    acc = _fill_bits(total, torch.float32, 0x7FC0BEEF)
    for t, s in enumerate(specs):
        o = db.offsets[t]
        grad[o:o + s.numel].copy_(grad_values(w, gi, t, device=DEV).reshape(-1))
        acc[o:o + s.numel].copy_(_acc_values(w, gi, t, s))
    g_h = host_bits(grad).copy()
    a_h = f32(acc).copy()
    norms, tot, flag = db.norm_nonfinite(grad)
    db.scale_accum_zero(grad, acc, w.scale)
    codes = scales = None
    if db.n_scales:
        codes = torch.full((total,), 0x5A, dtype=torch.uint8, device=DEV)
        codes, scales = db.block_quant(acc, codes=codes)
    torch.cuda.synchronize()

    wn, wt, wf = oracle_lib.norm_nonfinite(op, g_h)
    assert wf == 0 and int(flag.item()) == 0
    assert_norms_close(f32(norms), tot.item(), wn, wt, what=f"{w.key} norms")
    oracle_lib.scale_accum_zero(op, g_h, a_h, w.scale)
    _assert_raw_equal(_raw(acc), a_h.view(np.uint32), f"{w.key} accumulate (whole buffer)")
    _assert_raw_equal(_raw(grad), g_h.view(np.uint16 if g_h.dtype == np.uint16 else np.uint32),
                      f"{w.key} zero (whole buffer)")
    del grad, g_h
    if codes is not None:
        wc = np.full(total, 0x5A, np.uint8)
        ws = oracle_lib.block_quant(op, specs, a_h, wc)
        _assert_raw_equal(_raw(scales), ws.view(np.uint32), f"{w.key} scales")
        _assert_raw_equal(_raw(codes), wc, f"{w.key} codes (whole buffer)")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0
    db.close()
    del acc, codes, scales
    torch.cuda.empty_cache()


def test_dense7b_layer_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("dense7b")
    sampled_group_parity(oracle_lib, oracle_plans("dense7b", 0), w, 0,
                         list(range(len(w.groups[0].tensors))))


def test_dense7b_embedding_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("dense7b")
    sampled_group_parity(oracle_lib, oracle_plans("dense7b", 1), w, 1, [0])


def test_moe_group_full_size(dbuf_lib, oracle_lib, oracle_plans):
    """193 tensors, uneven local_units (shards of 1..4 units), bf16 gradients,
    INT8 1x128 blocks: whole buffers against the oracle's whole-group run."""
    whole_group_parity(oracle_lib, oracle_plans("moe", 0), workload("moe"), 0)


def test_mixed_group_full_size(dbuf_lib, oracle_lib, oracle_plans):
    """2000 tensors from 1 to 4M elements, m=32: whole buffers against the
    oracle's whole-group run."""
    whole_group_parity(oracle_lib, oracle_plans("mixed", 0), workload("mixed"), 0)


def test_tensor_beyond_32bit_offsets(dbuf_lib, oracle_lib):
    """One tensor of 2,149,580,800 elements (131200 x 16384, 128x128 E4M3 blocks)
    after a small vector, m=2: element offsets and indices past 2^31 in every
    operator of the step.  The layout against the oracle's plan; pack, unpack,
    scale/accumulate/zero and block quantisation bit for bit on sampled block
    rows (the first, the two on either side of the shard bound, the last); the
    norm of the whole tensor against the oracle's, taken in 1 GB pieces; the
    non-finite flag for one inf planted in the last element."""
    from fsdp_infra_gb300 import DBuffer, dbuf
    from workloads.configs import TensorSpec
    R, C, B = 131200, 16384, 128
    specs = [TensorSpec("lead", 1000, 1, 1),
             TensorSpec("huge", R, C, B, qblock=(B, B), quant="e4m3")]
    m, scale = 2, 0.5
    op = oracle_lib.plan_specs(specs, m, None, 16)
    db = DBuffer(specs, m, None, 16).upload()
    assert db.S == op.S and db.total == op.total
    assert db.offsets == [int(x) for x in op.offsets]
    assert db.shard_bounds == [int(x) for x in op.bounds]
    lo = db.offsets[1]
    n = specs[1].numel
    assert lo + n > 2 ** 31
    # the shard bound falls between two block rows of the large tensor
    cut = (db.S - lo) // C
    assert 0 < cut < R and (db.S - lo) % (B * C) == 0
    block_rows = sorted({0, cut // B - 1, cut // B, R // B - 1})

    gen = torch.Generator(device=DEV)
    gen.manual_seed(2024)
    lead = torch.randn(1000, 1, generator=gen, device=DEV) * 0.02
    huge = torch.randn(R, C, generator=gen, device=DEV) * 0.02
    buf16 = torch.zeros(db.total, dtype=torch.bfloat16, device=DEV)
    db.pack_cast([lead, huge], buf16)
    dst = [torch.empty(1000, 1, dtype=torch.bfloat16, device=DEV),
           torch.empty(R, C, dtype=torch.bfloat16, device=DEV)]
    db.unpack(buf16, dst)
    grad = torch.randn(db.total, generator=gen, device=DEV) * 1e-3
    acc = torch.randn(db.total, generator=gen, device=DEV) * 1e-3
    rows = [(b * B, (b + 1) * B) for b in block_rows]
    g_rows = [f32(grad[lo + r0 * C:lo + r1 * C]).copy() for r0, r1 in rows]
    a_rows = [f32(acc[lo + r0 * C:lo + r1 * C]).copy() for r0, r1 in rows]

    norms, tot, flag = db.norm_nonfinite(grad)
    torch.cuda.synchronize()
    # the oracle's norms: the vector whole, the large tensor in 2^28-element pieces
    # (sums of squares in fp64, recombined)
    sq = [float(oracle_lib.norm_nonfinite(oracle_lib.plan_specs([specs[0]], 1, None, 1),
                                          f32(grad[:1000]).copy())[0][0]) ** 2, 0.0]
    piece = 1 << 28
    for s0 in range(0, n, piece):
        k = min(piece, n - s0)
        sp = oracle_lib.plan_specs([TensorSpec("piece", k, 1, 1)], 1, None, 1)
        nn, _, wf = oracle_lib.norm_nonfinite(sp, f32(grad[lo + s0:lo + s0 + k]))
        assert wf == 0
        sq[1] += float(nn[0]) ** 2
    want = np.sqrt(np.array(sq))
    assert int(flag.item()) == 0
    assert_norms_close(f32(norms), tot.item(), want, math.sqrt(sum(sq)), what="2^31+ norms")

    db.scale_accum_zero(grad, acc, scale)
    codes, scales = db.block_quant(acc)
    torch.cuda.synchronize()
    so = int(oracle_lib.scale_offsets(specs)[0][1])
    nbc = C // B
    for (r0, r1), g_h, a_h in zip(rows, g_rows, a_rows):
        sub = TensorSpec("rows", r1 - r0, C, B, qblock=(B, B), quant="e4m3")
        sp = oracle_lib.plan_specs([sub], 1, None, 1)
        k = sub.numel
        base = lo + r0 * C
        want16 = np.zeros(k, np.uint16)
        oracle_lib.pack(sp, [f32(huge[r0:r1]).reshape(-1)], want16)
        assert_bits_equal(bf16_bits(buf16[base:base + k]), want16, f"pack rows {r0}")
        wd = np.zeros(k, np.uint16)
        oracle_lib.unpack(sp, want16, [wd])
        assert_bits_equal(bf16_bits(dst[1][r0:r1]).reshape(-1), wd, f"unpack rows {r0}")
        oracle_lib.scale_accum_zero(sp, g_h, a_h, scale)
        assert_bits_equal(f32(acc[base:base + k]), a_h, f"accumulate rows {r0}")
        assert_bits_equal(f32(grad[base:base + k]), g_h, f"zero rows {r0}")
        wc = np.zeros(k, np.uint8)
        ws = oracle_lib.block_quant(sp, [sub], a_h, wc)
        b = r0 // B
        assert_bits_equal(f32(scales[so + b * nbc:so + (b + 1) * nbc]), ws[:nbc], f"scales rows {r0}")
        assert_bits_equal(codes[base:base + k].cpu().numpy(), wc, f"codes rows {r0}")

    grad[lo + n - 1] = float("inf")
    _, _, flag = db.norm_nonfinite(grad)
    assert int(flag.item()) == 1
    assert dbuf.dbuf_device_status(db.handle) == 0
    db.close()
    del lead, huge, buf16, dst, grad, acc, codes, scales
    torch.cuda.empty_cache()


def test_next_rows_beyond_32bit_offsets(dbuf_lib, oracle_lib):
    """The next rows past 32-bit offsets, on one 131200 x 16384 tensor
    (2,149,580,800 elements) after a vector, m=2: 8-bit AdamW with 32x32 INT8
    blocks (the pipelined kernel) and fp32 AdamW bit for bit against the oracle
    on sampled block rows (both ends, either side of the shard bound), with
    clipping; gather of the tensor from the two shard slices and scatter back,
    compared with the flat buffer on the same rows."""
    from fsdp_infra_gb300 import DBuffer, dbuf
    from workloads.configs import TensorSpec
    R, C, B = 131200, 16384, 32
    specs = [TensorSpec("lead", 1000, 1, 1),
             TensorSpec("huge", R, C, B, qblock=(B, B), quant="int8")]
    m = 2
    op = oracle_lib.plan_specs(specs, m, None, 16)
    db = DBuffer(specs, m, None, 16).upload()
    assert db.offsets == [int(x) for x in op.offsets] and db.total == op.total
    lo, n = db.offsets[1], specs[1].numel
    assert lo + n > 2 ** 31
    cut = (db.S - lo) // C
    assert 0 < cut < R and (db.S - lo) % (B * C) == 0
    block_rows = sorted({0, cut // B - 1, cut // B, R // B - 1})
    rows = [(b * B, (b + 1) * B) for b in block_rows]
    nbc = C // B
    hp = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    b1, b2 = hp["betas"]
    step, max_norm, total = 3, 0.5, 0.75
    okw = dict(lr=hp["lr"], beta1=b1, beta2=b2, eps=hp["eps"], weight_decay=hp["weight_decay"],
               step=step, max_norm=max_norm, total_norm=total)

    gen = torch.Generator(device=DEV)
    gen.manual_seed(31)
    p = torch.randn(db.total, generator=gen, device=DEV) * 0.02
    g = torch.randn(db.total, generator=gen, device=DEV) * 1e-3
    st = db.new_adamw8_state()
    st["m_codes"].copy_(torch.randint(0, 256, (db.total,), generator=gen, device=DEV,
                                      dtype=torch.int32).to(torch.uint8))
    st["v_codes"].copy_(torch.randint(0, 256, (db.total,), generator=gen, device=DEV,
                                      dtype=torch.int32).to(torch.uint8))
    st["m_scales"].uniform_(1e-7, 1e-5, generator=gen)
    st["v_scales"].uniform_(1e-12, 1e-9, generator=gen)
    so = int(oracle_lib.scale_offsets(specs)[0][1])
    before = []
    for r0, r1 in rows:
        a, e = lo + r0 * C, lo + r1 * C
        s0, s1 = so + (r0 // B) * nbc, so + (r1 // B) * nbc
        before.append({k: x for k, x in (
            ("p", f32(p[a:e]).copy()), ("g", f32(g[a:e]).copy()),
            ("mc", st["m_codes"][a:e].cpu().numpy().copy()),
            ("vc", st["v_codes"][a:e].cpu().numpy().copy()),
            ("ms", f32(st["m_scales"][s0:s1]).copy()), ("vs", f32(st["v_scales"][s0:s1]).copy()))})
    tn = torch.tensor([total], dtype=torch.float32, device=DEV)
    db.adamw8_step(p, g, st, step=step, max_norm=max_norm, total_norm=tn, **hp)
    torch.cuda.synchronize()
    for (r0, r1), h in zip(rows, before):
        sub = TensorSpec("rows", r1 - r0, C, B, qblock=(B, B), quant="int8")
        sp = oracle_lib.plan_specs([sub], 1, None, 1)
        z = np.zeros(1, np.float32)
        oracle_lib.adamw8(sp, [sub], h["p"], h["g"], h["mc"], h["vc"], h["ms"], h["vs"], z,
                          z.copy(), **okw)
        a, e = lo + r0 * C, lo + r1 * C
        s0, s1 = so + (r0 // B) * nbc, so + (r1 // B) * nbc
        assert_bits_equal(f32(p[a:e]), h["p"], f"adamw8 params rows {r0}")
        assert np.array_equal(st["m_codes"][a:e].cpu().numpy(), h["mc"]), f"m codes rows {r0}"
        assert np.array_equal(st["v_codes"][a:e].cpu().numpy(), h["vc"]), f"v codes rows {r0}"
        assert_bits_equal(f32(st["m_scales"][s0:s1]), h["ms"], f"m scales rows {r0}")
        assert_bits_equal(f32(st["v_scales"][s0:s1]), h["vs"], f"v scales rows {r0}")
    del st
    torch.cuda.empty_cache()

    # fp32 AdamW on the same buffers
    mom = torch.randn(db.total, generator=gen, device=DEV) * 1e-4
    vel = torch.rand(db.total, generator=gen, device=DEV) * 1e-8
    before = []
    for r0, r1 in rows:
        a, e = lo + r0 * C, lo + r1 * C
        before.append([f32(x[a:e]).copy() for x in (p, g, mom, vel)])
    db.adamw_step(p, g, mom, vel, step=step, max_norm=max_norm, total_norm=tn, **hp)
    torch.cuda.synchronize()
    for (r0, r1), (hp_, hg, hm, hv) in zip(rows, before):
        sp = oracle_lib.plan_specs([TensorSpec("rows", r1 - r0, C, B)], 1, None, 1)
        oracle_lib.adamw(sp, hp_, hg, hm, hv, **okw)
        a, e = lo + r0 * C, lo + r1 * C
        assert_bits_equal(f32(p[a:e]), hp_, f"adamw params rows {r0}")
        assert_bits_equal(f32(mom[a:e]), hm, f"adamw m rows {r0}")
        assert_bits_equal(f32(vel[a:e]), hv, f"adamw v rows {r0}")
    del mom, vel
    torch.cuda.empty_cache()

    # gather from the two shard slices of p, scatter back into zeroed slices of g
    bnd = db.shard_bounds
    shards = [p[bnd[k]:bnd[k + 1]] for k in range(m)]
    full = torch.empty(R, C, dtype=torch.float32, device=DEV)
    db.gather(shards, [None, full])
    g.zero_()
    back = [g[bnd[k]:bnd[k + 1]] for k in range(m)]
    db.scatter([None, full], back)
    torch.cuda.synchronize()
    for r0, r1 in rows:
        a, e = lo + r0 * C, lo + r1 * C
        want = f32(p[a:e])
        assert_bits_equal(f32(full[r0:r1]).reshape(-1), want, f"gather rows {r0}")
        assert_bits_equal(f32(g[a:e]), want, f"scatter rows {r0}")
    assert float(g[:1000].abs().max().item()) == 0.0  # the skipped vector stays untouched
    assert dbuf.dbuf_device_status(db.handle) == 0
    db.close()
    del p, g, full, shards, back
    torch.cuda.empty_cache()
