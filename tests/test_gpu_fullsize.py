"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: the 7B-shaped dense layer and embedding DBuffers (m=64), the
MoE group (uneven local_units, bf16 grads, INT8 1x128) and the 2000-tensor mixed
group (m=32).  The layouts are compared whole; the operator outputs are compared
bit for bit on sampled tensors (every tensor for the dense groups), each checked
against the oracle run on that tensor alone; norms and the non-finite flag are
checked for every tensor.  Inputs are drawn on the device by torch's seeded
generator and copied to the host for the oracle.
"""
import math
import random

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


def test_dense7b_layer_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("dense7b")
    sampled_group_parity(oracle_lib, oracle_plans("dense7b", 0), w, 0,
                         list(range(len(w.groups[0].tensors))))


def test_dense7b_embedding_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("dense7b")
    sampled_group_parity(oracle_lib, oracle_plans("dense7b", 1), w, 1, [0])


def test_moe_group_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("moe")
    n = len(w.groups[0].tensors)
    sample = [0, 1, 2, 97, 98, 99, n - 3, n - 2, n - 1]
    sampled_group_parity(oracle_lib, oracle_plans("moe", 0), w, 0, sample)


def test_mixed_group_full_size(dbuf_lib, oracle_lib, oracle_plans):
    w = workload("mixed")
    specs = w.groups[0].tensors
    n = len(specs)
    rng = random.Random(4)
    by_size = sorted(range(n), key=lambda t: specs[t].numel)
    sample = sorted(set(rng.sample(range(n), 48) + by_size[:4] + by_size[-4:]))
    sampled_group_parity(oracle_lib, oracle_plans("mixed", 0), w, 0, sample)
