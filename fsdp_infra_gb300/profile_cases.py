"""Small launch cases for kernel captures: each runs one kind of launch a few
times on seeded synthetic buffers sized above L2 (129 MB) and a few GB on the
device at most, so that a counter capture of it ends in seconds.

    python -m fsdp_infra_gb300.profile_cases CASE [--reps R]

Cases:
  llama_step   every operator of the step and of the next rows once per rep on
               one Llama-style layer (51.4M elements, m=8, 128x128 E4M3):
               pack_cast, unpack, scale_accum_zero, norm_nonfinite, block_quant,
               adamw_step, adamw8_step (32x32 INT8 blocks), gather, scatter
  quant_row    block_quant on an MoE slice: 24 experts of the MoE group
               (gate/up 2048x1408, down 1408x2048; 207.6M elements, fp32
               accumulator 0.83 GB), row-wise units, INT8 1x128 blocks
  quant_tile   block_quant on the Llama layer over an fp32 buffer one element
               past a 16-byte boundary: every tile takes the register-tile kernel
  adamw8_big   adamw8_step on the Llama layer planned with 128x128 INT8 blocks
               (blocks of two pipeline stages: the big-block pipelined kernel)
  adamw8_reg   adamw8_step on the Llama layer planned with 128x96 INT8 blocks
               (not a power of two, so neither pipelined kernel takes them: the
               register kernel with its second pass over gradients and codes)
"""
from __future__ import annotations

import argparse
import sys

import torch

from .dbuffer import DBuffer


def _fill_ranges(db, buf, std, gen):
    for t, s in enumerate(db.specs):
        o = db.offsets[t]
        buf[o:o + s.rows * s.cols].normal_(0.0, std, generator=gen)


def _llama(block=None):
    from workloads import workload
    from workloads.configs import adam8_group
    w = workload("llama_layer")
    g = w.groups[0] if block is None else adam8_group(w.groups[0], block)
    return w, g


def case_llama_step(dev, reps):
    from workloads import param_values
    w, g = _llama()
    db = DBuffer(g.tensors, w.m, None, w.align, device=dev).upload()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    params = [param_values(w, 0, t, device=dev) for t in range(len(g.tensors))]
    compute = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=dev) for s in g.tensors]
    b16 = db.new_buffer(torch.bfloat16)
    grad, acc = db.new_buffer(torch.float32), db.new_buffer(torch.float32)
    _fill_ranges(db, grad, 1e-3, gen)
    codes = torch.zeros(db.total, dtype=torch.uint8, device=dev)
    p32, m32, v32 = (db.new_buffer(torch.float32) for _ in range(3))
    db.pack_cast(params, p32)
    _, g8 = _llama((32, 32))
    db8 = DBuffer(g8.tensors, w.m, None, w.align, device=dev).upload()
    p8, gg8 = db8.new_buffer(torch.float32), db8.new_buffer(torch.float32)
    _fill_ranges(db8, p8, 0.02, gen)
    _fill_ranges(db8, gg8, 1e-3, gen)
    st8 = db8.new_adamw8_state()
    shards = [acc[db.shard_bounds[k]:db.shard_bounds[k + 1]] for k in range(db.m)]
    mats = [torch.empty(s.rows * s.cols, dtype=torch.float32, device=dev) for s in g.tensors]
    for r in range(reps):
        db.pack_cast(params, b16)
        db.unpack(b16, compute)
        db.scale_accum_zero(grad, acc, w.scale)
        norms, total, flag = db.norm_nonfinite(acc)
        db.block_quant(acc, codes=codes)
        db.adamw_step(p32, acc, m32, v32, step=r + 1, lr=1e-4, betas=(0.9, 0.95),
                      weight_decay=0.1, max_norm=1.0, total_norm=total, nonfinite=flag)
        db8.adamw8_step(p8, gg8, st8, step=r + 1, lr=1e-4, betas=(0.9, 0.95), weight_decay=0.1)
        db.gather(shards, mats)
        db.scatter(mats, shards)
    return (f"llama_step: {reps} reps of the five step operators, AdamW, 8-bit AdamW, gather and "
            f"scatter on {sum(db.numel)} elements")


def case_quant_row(dev, reps):
    from workloads import workload
    from workloads.configs import GroupSpec
    w = workload("moe")
    ts = w.groups[0].tensors[:72]
    g = GroupSpec("moe24", tuple(ts))
    db = DBuffer(g.tensors, w.m, w.local_units, w.align, device=dev).upload()
    acc = db.new_buffer(torch.float32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2)
    _fill_ranges(db, acc, 1e-3, gen)
    codes = torch.zeros(db.total, dtype=torch.uint8, device=dev)
    for _ in range(reps):
        db.block_quant(acc, codes=codes)
    return f"quant_row: {reps} launches on {sum(db.numel)} elements, {db.n_scales} 1x128 blocks"


def case_quant_tile(dev, reps):
    w, g = _llama()
    db = DBuffer(g.tensors, w.m, None, w.align, device=dev).upload()
    raw = torch.zeros(db.total + 4, dtype=torch.float32, device=dev)
    acc = raw[1:1 + db.total]  # 4 bytes past a 16-byte boundary
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    _fill_ranges(db, acc, 1e-3, gen)
    codes = torch.zeros(db.total, dtype=torch.uint8, device=dev)
    for _ in range(reps):
        db.block_quant(acc, codes=codes)
    return f"quant_tile: {reps} launches on {sum(db.numel)} elements, unaligned fp32 buffer"


def _adamw8(dev, reps, block):
    w, g = _llama(block)
    db = DBuffer(g.tensors, w.m, None, w.align, device=dev).upload()
    p, gr = db.new_buffer(torch.float32), db.new_buffer(torch.float32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    _fill_ranges(db, p, 0.02, gen)
    _fill_ranges(db, gr, 1e-3, gen)
    st = db.new_adamw8_state()
    for r in range(reps):
        db.adamw8_step(p, gr, st, step=r + 1, lr=1e-4, betas=(0.9, 0.95), weight_decay=0.1)
    return sum(db.numel)


def case_adamw8_big(dev, reps):
    n = _adamw8(dev, reps, (128, 128))
    return f"adamw8_big: {reps} launches on {n} elements, 128x128 INT8 blocks"


def case_adamw8_reg(dev, reps):
    n = _adamw8(dev, reps, (128, 96))
    return f"adamw8_reg: {reps} launches on {n} elements, 128x96 INT8 blocks"


CASES = {"llama_step": case_llama_step, "quant_row": case_quant_row,
         "quant_tile": case_quant_tile, "adamw8_big": case_adamw8_big,
         "adamw8_reg": case_adamw8_reg}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    torch.cuda.set_device(0)
    msg = CASES[args.case](torch.device("cuda", 0), args.reps)
    torch.cuda.synchronize()
    print(msg, flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
