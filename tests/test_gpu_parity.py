"""GPU parity of every group operator against the oracle, through the C ABI.

Bit-exact: layout, pack/unpack (with the fp32->bf16 RNE cast), scale/accumulate/
zero, block-quantisation codes and scales.  Norms: within 1e-5 relative of the
oracle's fp64 norms (fp32 squares and sums against an fp64 reference).  Small
workloads are compared over whole buffers, padding included (padding must stay
exactly as it was).
"""
import math

import numpy as np
import pytest
import torch

from workloads import workload
from workloads.configs import TensorSpec, param_values, grad_values, inf_injection

from gpu_helpers import (assert_bits_equal, assert_norms_close, bf16_bits, f32, host_bits,
                         padding_mask)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lib(dbuf_lib):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    return dbuf_lib


def _db(specs, m, units=None, align=16):
    from fsdp_infra_gb300 import DBuffer
    return DBuffer(specs, m, units, align).upload()


def _check_layout(db, op):
    assert db.S == op.S and db.total == op.total
    assert db.offsets == [int(x) for x in op.offsets]
    assert db.shard_bounds == [int(x) for x in op.bounds]


def _sentinel_buffer(total, dtype, value):
    if dtype == torch.uint8:
        return torch.full((total,), value, dtype=torch.uint8, device=DEV)
    return torch.full((total,), value, dtype=dtype, device=DEV)


def full_group_parity(oracle_lib, specs, m, units, align, *, param_fn, grad_fn, grad_dtype,
                      scale, accum_steps=1, check_quant=True):
    """Run every operator on one group and compare whole buffers with the oracle."""
    op = oracle_lib.plan_specs(specs, m, units, align)
    db = _db(specs, m, units, align)
    _check_layout(db, op)
    n = len(specs)
    total = db.total
    numel = [s.numel for s in specs]
    pad = padding_mask(total, db.offsets, numel)

    # ---- pack fp32 -> fp32 and fp32 -> bf16; padding sentinel must survive
    params = [param_fn(t) for t in range(n)]
    src = [p.to(DEV).contiguous() for p in params]
    buf32 = _sentinel_buffer(total, torch.float32, 7.0)
    buf16 = _sentinel_buffer(total, torch.bfloat16, 7.0)
    db.pack_cast(src, buf32)
    db.pack_cast(src, buf16)
    want32 = np.full(total, 7.0, np.float32)
    want16 = np.full(total, bf16_bits(torch.tensor([7.0], dtype=torch.bfloat16))[0], np.uint16)
    host_src = [f32(p) for p in params]
    oracle_lib.pack(op, host_src, want32)
    oracle_lib.pack(op, host_src, want16)
    assert_bits_equal(f32(buf32), want32, "pack f32->f32")
    assert_bits_equal(bf16_bits(buf16), want16, "pack f32->bf16")

    # ---- unpack bf16 -> bf16, f32 -> f32, bf16 -> f32, f32 -> bf16
    for bsrc, bwant, ddt in [(buf16, want16, torch.bfloat16), (buf32, want32, torch.float32),
                             (buf16, want16, torch.float32), (buf32, want32, torch.bfloat16)]:
        dst = [torch.empty(s.rows, s.cols, dtype=ddt, device=DEV) for s in specs]
        db.unpack(bsrc, dst)
        hdst = [np.zeros(s.numel, np.float32 if ddt == torch.float32 else np.uint16) for s in specs]
        oracle_lib.unpack(op, bwant, hdst)
        for t in range(n):
            assert_bits_equal(host_bits(dst[t]).reshape(-1), hdst[t], f"unpack tensor {t} {bsrc.dtype}->{ddt}")

    # ---- scale / accumulate / zero over accum_steps steps
    gen = torch.Generator().manual_seed(99)
    acc0 = (torch.randn(total, generator=gen) * 1e-3).to(torch.float32)
    acc = acc0.to(DEV)
    acc_h = f32(acc0).copy()
    grad = _sentinel_buffer(total, grad_dtype, -3.0)
    for step in range(accum_steps):
        gvals = [grad_fn(t, step) for t in range(n)]
        for t, g in enumerate(gvals):
            grad[db.offsets[t]:db.offsets[t] + numel[t]].copy_(g.reshape(-1).to(DEV))
        g_h = host_bits(grad)
        db.scale_accum_zero(grad, acc, scale)
        oracle_lib.scale_accum_zero(op, g_h, acc_h, scale)
        assert_bits_equal(host_bits(grad), g_h, f"grad zeroed step {step}")
        assert_bits_equal(f32(acc), acc_h, f"accumulator step {step}")

    # ---- norms + non-finite flag on the accumulator (fp32) and a bf16 buffer
    norms, tot, flag = db.norm_nonfinite(acc)
    wn, wt, wf = oracle_lib.norm_nonfinite(op, acc_h)
    assert int(flag.item()) == wf == 0
    assert_norms_close(f32(norms), tot.item(), wn, wt, what="norm fp32")
    norms, tot, flag = db.norm_nonfinite(buf16)
    wn, wt, wf = oracle_lib.norm_nonfinite(op, want16)
    assert int(flag.item()) == wf
    assert_norms_close(f32(norms), tot.item(), wn, wt, what="norm bf16")

    # ---- block quantisation of the accumulator
    if check_quant and any(s.quant for s in specs):
        codes = _sentinel_buffer(total, torch.uint8, 0xAB)
        codes, scales = db.block_quant(acc, codes=codes)
        want_codes = np.full(total, 0xAB, np.uint8)
        want_scales = oracle_lib.block_quant(op, specs, acc_h, want_codes)
        assert db.n_scales == want_scales.size
        assert_bits_equal(f32(scales), want_scales, "scales")
        assert_bits_equal(codes.cpu().numpy(), want_codes, "codes")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0
    return db, op


def _workload_fns(w, gi=0):
    return (lambda t: param_values(w, gi, t),
            lambda t, step: grad_values(w, gi, t, step=step))


def test_tiny_transformer_group(lib, oracle_lib):
    w = workload("tiny")
    pf, gf = _workload_fns(w)
    full_group_parity(oracle_lib, w.groups[0].tensors, w.m, w.local_units, w.align,
                      param_fn=pf, grad_fn=gf, grad_dtype=w.grad_dtype, scale=w.scale)


@pytest.mark.parametrize("m", [64, 1024])
def test_tiny_group_at_high_shard_counts(lib, oracle_lib, m):
    """The tiny group over 64 and 1024 shards (most of them padding only): every
    operator on whole buffers against the oracle."""
    w = workload("tiny")
    pf, gf = _workload_fns(w)
    full_group_parity(oracle_lib, w.groups[0].tensors, m, None, w.align,
                      param_fn=pf, grad_fn=gf, grad_dtype=w.grad_dtype, scale=1.0 / m)


def test_llama_layer_accumulation(lib, oracle_lib):
    w = workload("llama_layer")
    pf, gf = _workload_fns(w)
    full_group_parity(oracle_lib, w.groups[0].tensors, w.m, w.local_units, w.align,
                      param_fn=pf, grad_fn=gf, grad_dtype=w.grad_dtype, scale=w.scale,
                      accum_steps=w.accum_steps)


def test_llama_layer_inf_injection_runs(lib, oracle_lib, oracle_plans):
    """Ten gradient runs; one carries a single +inf: only that run raises the flag."""
    w = workload("llama_layer")
    specs = w.groups[0].tensors
    op = oracle_plans("llama_layer", 0)
    db = _db(specs, w.m, None, w.align)
    r_inf, t_inf, i_inf = inf_injection(w, runs=10)
    grad = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    for run in range(10):
        for t in range(len(specs)):
            g = grad_values(w, 0, t, seed=run, device=DEV).reshape(-1)
            if run == r_inf and t == t_inf:
                g[i_inf] = float("inf")
            grad[db.offsets[t]:db.offsets[t] + specs[t].numel].copy_(g)
        norms, tot, flag = db.norm_nonfinite(grad)
        gh = f32(grad)
        wn, wt, wf = oracle_lib.norm_nonfinite(op, gh)
        assert int(flag.item()) == wf == (1 if run == r_inf else 0)
        if wf == 0:
            assert_norms_close(f32(norms), tot.item(), wn, wt)


def test_uneven_local_units_rowwise_int8(lib, oracle_lib):
    """A small MoE-shaped group: row-wise RaggedShard, uneven shares, bf16 grads,
    INT8 1x128 blocks including a partial 1x64 block per row."""
    specs = []
    for e in range(3):
        specs += [TensorSpec(f"e{e}.gate", 64, 176, 1, (1, 128), "int8"),
                  TensorSpec(f"e{e}.down", 176, 64, 1, (1, 128), "int8")]
    specs.append(TensorSpec("router", 64, 8, 1, (1, 128), "int8"))
    gen = torch.Generator().manual_seed(3)
    ps = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    gs = [[(torch.randn(s.rows, s.cols, generator=gen) * 1e-3).to(torch.bfloat16) for s in specs]
          for _ in range(2)]
    full_group_parity(oracle_lib, specs, 4, [1, 3, 2, 4], 16,
                      param_fn=lambda t: ps[t], grad_fn=lambda t, k: gs[k][t],
                      grad_dtype=torch.bfloat16, scale=1.0 / 4, accum_steps=2)


def test_ragged_edges_and_generic_paths(lib, oracle_lib):
    """Sizes off every vector width, tensors smaller than a unit, an empty tensor,
    quantisation tiles with partial rows/columns, odd widths (scalar path),
    blocks wider than 128 columns, and E4M3 and INT8 tensors in one group."""
    specs = [
        TensorSpec("v1", 1, 1, 1),
        TensorSpec("odd", 37, 3, 1),
        TensorSpec("empty", 0, 8, 1),
        TensorSpec("tile", 200, 136, 128, (128, 128), "e4m3"),
        TensorSpec("oddq", 130, 7, 0, (128, 128), "e4m3"),
        TensorSpec("wide", 40, 300, 0, (8, 256), "e4m3"),
        TensorSpec("rows", 33, 100, 1, (1, 32), "int8"),
        TensorSpec("rows_odd", 5, 129, 1, (1, 128), "int8"),
        TensorSpec("big", 3 * 16384 + 13, 1, 1),
    ]
    gen = torch.Generator().manual_seed(11)
    ps = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    gs = [torch.randn(s.rows, s.cols, generator=gen) * 1e-3 for s in specs]
    for m, align in [(3, 16), (1, 16), (5, 1), (7, 4)]:
        full_group_parity(oracle_lib, specs, m, None, align,
                          param_fn=lambda t: ps[t], grad_fn=lambda t, k: gs[t],
                          grad_dtype=torch.float32, scale=0.3)


def test_misaligned_user_tensors_take_scalar_path(lib, oracle_lib):
    """User tensors at odd element offsets (not 16-byte aligned) give the same
    bytes as the vector path."""
    specs = [TensorSpec("a", 100, 33, 1), TensorSpec("b", 4097, 1, 1)]
    op = oracle_lib.plan_specs(specs, 2, None, 16)
    db = _db(specs, 2)
    gen = torch.Generator().manual_seed(5)
    base = [torch.randn(s.numel + 1, generator=gen).to(DEV) for s in specs]
    src = [b[1:] for b in base]                      # offset by one fp32 element
    buf = torch.zeros(db.total, dtype=torch.bfloat16, device=DEV)
    db.pack_cast(src, buf)
    want = np.zeros(db.total, np.uint16)
    oracle_lib.pack(op, [f32(s) for s in src], want)
    assert_bits_equal(bf16_bits(buf), want, "pack from misaligned sources")
    dst_base = [torch.zeros(s.numel + 1, dtype=torch.float32, device=DEV) for s in specs]
    dst = [d[1:] for d in dst_base]
    db.unpack(buf, dst)
    hd = [np.zeros(s.numel, np.float32) for s in specs]
    oracle_lib.unpack(op, want, hd)
    for t in range(2):
        assert_bits_equal(f32(dst[t]), hd[t], "unpack to misaligned destinations")


def test_cast_special_values(lib, oracle_lib):
    """fp32->bf16 on the GPU vs the oracle over every upper half-word with the
    rounding-critical lower halves, plus signed zeros and infinities; NaN stays
    NaN."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    bits = np.concatenate([hi | lo for lo in (0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF)])
    x = bits.view(np.float32)
    specs = [TensorSpec("x", x.size, 1, 1)]
    op = oracle_lib.plan_specs(specs, 1, None, 16)
    db = _db(specs, 1)
    buf = torch.zeros(db.total, dtype=torch.bfloat16, device=DEV)
    db.pack_cast([torch.from_numpy(x).to(DEV)], buf)
    want = np.zeros(db.total, np.uint16)
    oracle_lib.pack(op, [x], want)
    got = bf16_bits(buf)
    gf = (got.astype(np.uint32) << 16).view(np.float32)
    wf = (want.astype(np.uint32) << 16).view(np.float32)
    nan = np.isnan(wf)
    assert np.array_equal(np.isnan(gf), nan)
    assert_bits_equal(got[~nan], want[~nan], "bf16 cast")


def test_fp8_and_int8_encoding_sweep(lib, oracle_lib):
    """With a block amax of exactly qmax the scale is 1.0, so the codes are the
    plain encodings of the inputs: compares the GPU encoders with the oracle's over
    ties, subnormals and saturation."""
    mags = np.array([oracle_lib.e4m3_value(c) for c in range(127)])
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mags.astype(np.float32), mids, np.nextafter(mids, np.float32(1e9)),
                           np.nextafter(mids, np.float32(0)),
                           np.linspace(0, 448, 4096, dtype=np.float32), [2.0 ** -12, 1e-30]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    cols = 128
    rows = -(-vals.size // cols)
    x = np.zeros(rows * cols, np.float32)
    x[:vals.size] = vals
    x = x.reshape(rows, cols)
    halves = np.arange(-126.5, 127.0, 0.5, dtype=np.float32)       # exact ties included
    rnd = np.random.default_rng(8).uniform(-127, 127, rows * cols - halves.size).astype(np.float32)
    xi = np.concatenate([halves, rnd]).reshape(rows, cols)
    for q, qmax, qb in [("e4m3", 448.0, (rows, cols)), ("int8", 127.0, (1, cols))]:
        y = x.copy() if q == "e4m3" else xi.copy()
        y[0, 0] = qmax  # every block has amax == qmax -> scale 1.0
        if q == "int8":
            y[:, 0] = qmax
        specs = [TensorSpec("w", rows, cols, 0, qb, q)]
        op = oracle_lib.plan_specs(specs, 1, None, 16)
        db = _db(specs, 1)
        buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
        buf[:y.size].copy_(torch.from_numpy(y.reshape(-1)))
        codes, scales = db.block_quant(buf)
        wc = np.zeros(db.total, np.uint8)
        ws = oracle_lib.block_quant(op, specs, f32(buf), wc)
        assert np.all(ws == 1.0)
        assert_bits_equal(f32(scales), ws, f"{q} scales")
        assert_bits_equal(codes.cpu().numpy(), wc, f"{q} codes")


def test_empty_group(lib):
    db = _db([], 4)
    assert db.total == 0
    buf = torch.zeros(16, dtype=torch.float32, device=DEV)
    db.pack_cast([], buf)
    norms, tot, flag = db.norm_nonfinite(buf)
    assert tot.item() == 0.0 and flag.item() == 0


def test_group_of_empty_tensors(lib, oracle_lib):
    """Tensors that all have no element (a plan of total 0, flat buffers of no
    element, whose device pointers are NULL): every operator accepts the call,
    touches nothing, and the norms are zero with the flag clear."""
    specs = [TensorSpec("q", 0, 158, 1, qblock=(1, 128), quant="e4m3"),
             TensorSpec("v", 0, 1, 1), TensorSpec("t", 0, 10, 5, qblock=(5, 4), quant="int8")]
    for m, units in ((8, None), (4, [4, 1, 4, 3])):
        db = _db(specs, m, units, 1)
        assert db.total == 0
        empty = torch.zeros(0, dtype=torch.float32, device=DEV)
        e16 = torch.zeros(0, dtype=torch.bfloat16, device=DEV)
        users = [torch.zeros(s.rows, s.cols, dtype=torch.float32, device=DEV) for s in specs]
        db.pack_cast(users, e16)
        db.unpack(e16, users)
        db.scale_accum_zero(empty, empty, 0.5)
        norms, tot, flag = db.norm_nonfinite(empty)
        assert norms[:3].tolist() == [0.0, 0.0, 0.0] and tot.item() == 0.0 and flag.item() == 0
        codes, scales = db.block_quant(empty, codes=torch.zeros(0, dtype=torch.uint8, device=DEV))
        assert codes.numel() == 0 and scales.numel() == 0
        db.adamw_step(empty, empty, empty, empty, step=1, lr=1e-3)
        db.adamw8_step(empty, empty, db.new_adamw8_state(), step=1, lr=1e-3)
        shards = [torch.zeros(0, dtype=torch.float32, device=DEV) for _ in range(m)]
        mats = [torch.zeros(0, dtype=torch.float32, device=DEV) for _ in specs]
        db.gather(shards, mats)
        db.scatter(mats, shards)
        from fsdp_infra_gb300 import dbuf
        assert dbuf.dbuf_device_status(db.handle) == 0
        db.close()


def test_norm_is_deterministic_and_flags_nan(lib, oracle_lib):
    w = workload("tiny")
    specs = w.groups[0].tensors
    db = _db(specs, w.m)
    buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    for t in range(len(specs)):
        buf[db.offsets[t]:db.offsets[t] + specs[t].numel].copy_(
            grad_values(w, 0, t, device=DEV).reshape(-1))
    a = [x.clone() for x in db.norm_nonfinite(buf)]
    b = db.norm_nonfinite(buf)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    # NaN in a tensor range raises the flag; a NaN in the padding does not.
    o = db.offsets[3] + 17
    buf[o] = float("nan")
    assert db.norm_nonfinite(buf)[2].item() == 1
    buf[o] = 0.0
    pad = padding_mask(db.total, db.offsets, [s.numel for s in specs])
    idx = np.nonzero(pad)[0]
    if idx.size:
        buf[int(idx[0])] = float("inf")
        assert db.norm_nonfinite(buf)[2].item() == 0


def test_all_ones_norm_is_exact(lib):
    specs = [TensorSpec("a", 64, 64, 1), TensorSpec("b", 16384 * 4, 1, 1)]
    db = _db(specs, 2)
    buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    for t, s in enumerate(specs):
        buf[db.offsets[t]:db.offsets[t] + s.numel] = 1.0
    norms, tot, flag = db.norm_nonfinite(buf)
    assert norms.tolist() == [64.0, 256.0]
    assert tot.item() == pytest.approx(math.sqrt(4096 + 65536), rel=1e-7)


def test_operators_on_a_side_stream(lib, oracle_lib):
    w = workload("tiny")
    specs = w.groups[0].tensors
    op = oracle_lib.plan_specs(specs, w.m, None, w.align)
    db = _db(specs, w.m)
    src = [param_values(w, 0, t).to(DEV) for t in range(len(specs))]
    buf = torch.zeros(db.total, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        db.pack_cast(src, buf, stream=s)
    s.synchronize()
    want = np.zeros(db.total, np.uint16)
    oracle_lib.pack(op, [f32(x) for x in src], want)
    assert_bits_equal(bf16_bits(buf), want, "pack on a side stream")


def test_quant_quotient_stress(lib, oracle_lib):
    """Blocks whose scales straddle 2^-80 (below it the kernel divides with the
    IEEE instructions, above it from the block's reciprocal), subnormal and
    signed-zero inputs, and inputs whose quotient by a non-trivial scale sits on
    or next to an E4M3 midpoint or an INT8 half-integer."""
    rng = np.random.default_rng(21)
    mags = np.array([oracle_lib.e4m3_value(c) for c in range(127)])
    mids = (mags[:-1] + mags[1:]) / 2
    rows, cols = 64, 128
    blocks = []
    for amax in [1e-38, 2.0 ** -70 * 448, 2.0 ** -80 * 448 * 0.999, 2.0 ** -80 * 448 * 1.001,
                 3.1e-3, 0.02, 1.7, 123.0, 3e30]:
        for q, qmax, targets in [("e4m3", 448.0, mids), ("int8", 127.0,
                                                         np.arange(-126.5, 127.0, 1.0))]:
            s = np.float32(np.float32(amax) / np.float32(qmax))
            t = rng.choice(targets, rows * cols)
            x = (t * np.float64(s)).astype(np.float32)
            k = rng.integers(-2, 3, x.size)
            x = np.array([np.float32(v) if d == 0 else
                          (np.nextafter(v, np.float32(np.inf * np.sign(d))) if abs(d) == 1 else
                           np.nextafter(np.nextafter(v, np.float32(np.inf * np.sign(d))),
                                        np.float32(np.inf * np.sign(d))))
                          for v, d in zip(x, k)], np.float32)
            x[:16] = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-40, -3e-39, 2e-38, -2e-38] * 2,
                              np.float32)
            x = np.clip(x, -np.float32(amax), np.float32(amax))
            x[16] = np.float32(amax)          # fixes the block's amax
            blocks.append((q, x.reshape(rows, cols)))
    for q in ("e4m3", "int8"):
        data = [b for kind, b in blocks if kind == q]
        qb = (rows, cols) if q == "e4m3" else (1, cols)
        specs = [TensorSpec(f"b{i}", rows, cols, 0, qb, q) for i in range(len(data))]
        op = oracle_lib.plan_specs(specs, 2, None, 16)
        db = _db(specs, 2)
        buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
        for i, x in enumerate(data):
            buf[db.offsets[i]:db.offsets[i] + x.size].copy_(torch.from_numpy(x.reshape(-1)))
        codes = torch.full((db.total,), 0xAB, dtype=torch.uint8, device=DEV)
        codes, scales = db.block_quant(buf, codes=codes)
        wc = np.full(db.total, 0xAB, np.uint8)
        ws = oracle_lib.block_quant(op, specs, f32(buf), wc)
        assert_bits_equal(f32(scales), ws, f"{q} stress scales")
        assert_bits_equal(codes.cpu().numpy(), wc, f"{q} stress codes")


def test_quant_unaligned_buffers_and_status(lib, oracle_lib):
    """Buffers that are not 16-byte aligned (fp32 input offset by one element,
    codes offset by one byte) cannot stream rows by bulk copy: the register-tile
    path must give the same codes; the device status stays clear."""
    specs = [TensorSpec("a", 256, 384, 128, (128, 128), "e4m3"),
             TensorSpec("v", 100, 1, 1),
             TensorSpec("b", 200, 136, 128, (128, 128), "int8")]
    op = oracle_lib.plan_specs(specs, 2, None, 16)
    db = _db(specs, 2)
    gen = torch.Generator().manual_seed(17)
    host = (torch.randn(db.total, generator=gen) * 0.05).to(torch.float32)
    want_c = np.full(db.total, 0x5A, np.uint8)
    want_s = oracle_lib.block_quant(op, specs, host.numpy().copy(), want_c)
    for fshift, cshift in [(0, 0), (1, 0), (0, 1), (1, 3)]:
        fb = torch.zeros(db.total + 4, dtype=torch.float32, device=DEV)
        fb[fshift:fshift + db.total].copy_(host)
        cb = torch.full((db.total + 4,), 0x5A, dtype=torch.uint8, device=DEV)
        codes, scales = db.block_quant(fb[fshift:fshift + db.total],
                                       codes=cb[cshift:cshift + db.total])
        assert_bits_equal(f32(scales), want_s, f"scales shift {fshift},{cshift}")
        assert_bits_equal(codes.cpu().numpy(), want_c, f"codes shift {fshift},{cshift}")
    assert lib.dbuf_device_status(db.handle) == 0


def test_quant_pipe_odd_block_rows(lib, oracle_lib):
    """Blocks of the pipelined tile kernel whose row count is odd or small (each
    half of a tile covers ceil(qrows / 2) rows, the second half one row short or
    empty), narrow blocks, ragged tensor edges, E4M3 and INT8: codes and scales
    bit-exact against the oracle on the whole buffer.  Every tensor qualifies
    for the tensor-map path: block widths and row lengths multiples of 4
    elements, offsets aligned to 16 elements."""
    specs = []
    for i, (qb, rows, cols) in enumerate([((7, 16), 23, 52), ((33, 64), 70, 200),
                                          ((127, 128), 300, 260), ((3, 4), 10, 20),
                                          ((2, 8), 9, 40), ((128, 96), 130, 100)]):
        quant = "e4m3" if i % 2 == 0 else "int8"
        specs.append(TensorSpec(f"w{i}", rows, cols, qb[0], qblock=qb, quant=quant))
    db = _db(specs, 2)
    op = oracle_lib.plan_specs(specs, 2, None, 16)
    gen = torch.Generator().manual_seed(23)
    host = (torch.randn(db.total, generator=gen) * 0.05).to(torch.float32)
    want_c = np.full(db.total, 0x5A, np.uint8)
    want_s = oracle_lib.block_quant(op, specs, host.numpy().copy(), want_c)
    cb = torch.full((db.total,), 0x5A, dtype=torch.uint8, device=DEV)
    codes, scales = db.block_quant(host.to(DEV), codes=cb)
    assert_bits_equal(f32(scales), want_s, "scales")
    assert_bits_equal(codes.cpu().numpy(), want_c, "codes")
    assert lib.dbuf_device_status(db.handle) == 0


def test_quant_more_tensors_than_one_launch_holds(lib, oracle_lib):
    """75 tensors of the pipelined quantisation kernel (three launches of at most
    32 tensors, block shapes 128x128, 64x128 and 32x32 in E4M3 and INT8 changing
    across the batch boundaries, ragged edges) with vectors between them; every
    operator against the oracle on whole buffers."""
    from workloads.configs import TensorSpec
    specs = []
    for i in range(75):
        qb = [(128, 128), (64, 128), (32, 32)][i % 3]
        quant = "e4m3" if i % 2 == 0 else "int8"
        rows = qb[0] * (1 + i % 3) + (5 if i % 4 == 1 else 0)
        cols = 128 * (1 + i % 2) + (64 if i % 5 == 2 else 0)
        specs.append(TensorSpec(f"w{i}", rows, cols, qb[0], qblock=qb, quant=quant))
        if i % 9 == 4:
            specs.append(TensorSpec(f"n{i}", 64 + i, 1, 1))
    gen = torch.Generator().manual_seed(17)
    ps = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    full_group_parity(oracle_lib, specs, 4, None, 16,
                      param_fn=lambda t: ps[t],
                      grad_fn=lambda t, step: torch.randn(specs[t].rows, specs[t].cols,
                                                          generator=gen) * 1e-3,
                      grad_dtype=torch.float32, scale=0.25)
