#!/usr/bin/env python3
"""Benchmark of the DBuffer group-operator pass on GB300.

One step = one pass of every group operator over every DBuffer of the 7B-shaped
dense stack (32 transformer layers d=4096 ffn=11008 + the 32000x4096 embedding,
one DBuffer per layer, m=64 shard slices, 128x128 blocks, E4M3 128x128 block
quantisation, s = 1/64): per DBuffer
  pack_cast  fp32 master params -> bf16 flat buffer      (6 B/elem)
  unpack     bf16 flat buffer -> bf16 compute tensors    (4 B/elem)
  scale_accum_zero  fp32 grads -> fp32 accumulator       (16 B/elem)
  norm_nonfinite    fp32 accumulator                     (4 B/elem)
  block_quant       fp32 accumulator -> E4M3 codes       (5 B/elem + 4 B/block)
Throughput = algorithmic bytes (tensor ranges only, padding excluded) / time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--exchange]
N>1 runs under torch.distributed.run: one independent replica per GPU (the path
has no exchange step on one GPU), timing max over ranks.  --exchange instead runs
the sharded step with its collectives, each DBuffer planned with m = N.  --impl
reference times the CPU oracle on a bounded sample of the same workload (rank 0
only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "fused group-op HBM GB/s (fraction of GB300 peak); params/sec per buffer pass"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
REF_SAMPLE_ROWS = 8000  # rows of the embedding table in the CPU sample


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (the slowest rank's time); x itself
    when not distributed."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job GB/s: every rank (one independent replica per GPU) moves
    bytes_per_rank_step per step; the step time is the slowest rank's."""
    return world * bytes_per_rank_step / (ms_per_step / 1e3) / 1e9


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                if self.uuid and self.uuid.replace("GPU-", "") not in p[0]:
                    continue
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload: every DBuffer of the 7B-shaped stack
# ---------------------------------------------------------------------------
def op_bytes_per_elem(grad_dtype):
    """Algorithmic bytes per element of each operator in the step (padding is
    never touched): pack_cast reads fp32 and writes bf16; unpack reads and writes
    bf16; scale_accum_zero reads the gradient and the fp32 accumulator, writes
    both; norm_nonfinite reads the fp32 accumulator.  block_quant (5 B/elem plus
    4 B per block scale) is counted per quantised element separately."""
    g = 2 if grad_dtype == torch.bfloat16 else 4
    return {"pack_cast": 6, "unpack": 4, "scale_accum_zero": 2 * g + 8, "norm_nonfinite": 4}


class Stack:
    """Plans, user tensors and flat buffers of the dense stack on one GPU.  The
    32 layer DBuffers share one plan and one set of flat buffers (the buffers are
    the padded m*S layout, 7.5x a layer, so one set is reused layer by layer);
    each DBuffer keeps its own user tensors."""

    def __init__(self, w, device, layers=None):
        from fsdp_infra_gb300 import DBuffer
        from workloads import param_values
        self.w = w
        self.device = device
        self.groups = []  # (group index, DBuffer, count)
        self.dbufs = []
        for gi, g in enumerate(w.groups):
            db = DBuffer(g.tensors, w.m, w.local_units, w.align, device=device).upload()
            kind = {"db": db, "gi": gi, "spec": g,
                    "buf16": torch.zeros(db.total, dtype=torch.bfloat16, device=device),
                    "grad": torch.zeros(db.total, dtype=w.grad_dtype, device=device),
                    "acc": torch.zeros(db.total, dtype=torch.float32, device=device),
                    "codes": torch.zeros(db.total, dtype=torch.uint8, device=device),
                    "scales": torch.zeros(max(db.n_scales, 1), dtype=torch.float32, device=device)}
            gen = torch.Generator(device=device)
            gen.manual_seed(1234 + gi)
            for t, s in enumerate(g.tensors):
                o = db.offsets[t]
                kind["grad"][o:o + s.numel].normal_(0.0, w.grad_std, generator=gen)
            reps = g.repeat if layers is None else min(g.repeat, layers)
            for r in range(reps):
                params = [param_values(w, gi, t, device=device, seed=1000 * r + gi)
                          for t in range(len(g.tensors))]
                compute = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=device)
                           for s in g.tensors]
                out = (torch.empty(len(g.tensors), dtype=torch.float32, device=device),
                       torch.empty(1, dtype=torch.float32, device=device),
                       torch.empty(1, dtype=torch.int32, device=device))
                db.ptr_table(params)
                db.ptr_table(compute)
                self.dbufs.append({"kind": kind, "params": params, "compute": compute,
                                   "out": out})
        self.elements = sum(g.numel * (g.repeat if layers is None else min(g.repeat, layers))
                            for g in w.groups)
        self.per_elem = op_bytes_per_elem(w.grad_dtype)
        self.op_bytes = {k: v * self.elements for k, v in self.per_elem.items()}
        qe, ns = 0, 0
        for d in self.dbufs:
            k = d["kind"]
            qe += sum(s.numel for s in k["spec"].tensors if s.quant)
            ns += k["db"].n_scales
        self.op_bytes["block_quant"] = 5 * qe + 4 * ns
        self.bytes_per_step = sum(self.op_bytes.values())
        # per DBuffer: one launch each for pack_cast, unpack and scale_accum_zero,
        # two for norm_nonfinite (the partials, then the finishing launch), and the
        # quantisation kernels: one launch per 32 tile-quantised tensors (the
        # tensor maps one launch carries) and one for row blocks
        self.launches_per_step = 0
        for d in self.dbufs:
            spec = d["kind"]["spec"]
            q = [s for s in spec.tensors if s.quant and s.numel]
            tiles = sum(1 for s in q if (s.qblock[0] or s.rows) > 1)
            rows = len(q) - tiles
            self.launches_per_step += 5 + (tiles + 31) // 32 + (1 if rows else 0)

    def run_op(self, op):
        """One operator alone over every DBuffer of the step, launched back to back."""
        w = self.w
        for d in self.dbufs:
            k, db = d["kind"], d["kind"]["db"]
            if op == "pack_cast":
                db.pack_cast(d["params"], k["buf16"])
            elif op == "unpack":
                db.unpack(k["buf16"], d["compute"])
            elif op == "scale_accum_zero":
                db.scale_accum_zero(k["grad"], k["acc"], w.scale)
            elif op == "norm_nonfinite":
                db.norm_nonfinite(k["acc"], out=d["out"])
            elif op == "block_quant":
                db.block_quant(k["acc"], codes=k["codes"], scales=k["scales"])
            else:
                raise ValueError(op)

    def step(self, timers=None):
        w = self.w
        for d in self.dbufs:
            k, db = d["kind"], d["kind"]["db"]
            if timers:
                timers.mark("pack_cast", 0)
            db.pack_cast(d["params"], k["buf16"])
            if timers:
                timers.mark("pack_cast", 1); timers.mark("unpack", 0)
            db.unpack(k["buf16"], d["compute"])
            if timers:
                timers.mark("unpack", 1); timers.mark("scale_accum_zero", 0)
            db.scale_accum_zero(k["grad"], k["acc"], w.scale)
            if timers:
                timers.mark("scale_accum_zero", 1); timers.mark("norm_nonfinite", 0)
            db.norm_nonfinite(k["acc"], out=d["out"])
            if timers:
                timers.mark("norm_nonfinite", 1); timers.mark("block_quant", 0)
            db.block_quant(k["acc"], codes=k["codes"], scales=k["scales"])
            if timers:
                timers.mark("block_quant", 1)


class RawEvent:
    """A CUDA timing event recorded with cudaEventRecordExternal, so that inside a
    stream capture it becomes a timestamp node of the graph (a plain record there
    only marks a dependency).  Uses the CUDA runtime PyTorch already loaded."""
    _rt = None

    @classmethod
    def rt(cls):
        if cls._rt is None:
            import ctypes
            rt = ctypes.CDLL("libcudart.so.13")
            rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
            rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
            rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                ctypes.c_void_p]
            rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]
            cls._rt = rt
        return cls._rt

    def __init__(self):
        import ctypes
        self.h = ctypes.c_void_p()
        assert self.rt().cudaEventCreate(ctypes.byref(self.h)) == 0

    def record(self, stream):
        assert self.rt().cudaEventRecordWithFlags(self.h, stream.cuda_stream, 1) == 0

    def elapsed_time(self, end):
        import ctypes
        ms = ctypes.c_float()
        assert self.rt().cudaEventElapsedTime(ctypes.byref(ms), self.h, end.h) == 0
        return ms.value

    def __del__(self):
        try:
            self.rt().cudaEventDestroy(self.h)
        except Exception:
            pass


class OpTimers:
    """CUDA events around operator launches on the launching stream (all
    operators, or only `only`); raw external events work inside graph capture."""

    def __init__(self, only=None, raw=False):
        self.only = only
        self.raw = raw
        self.events = {}

    def mark(self, op, which):
        if self.only is not None and op != self.only:
            return
        st = torch.cuda.current_stream()
        if self.raw:
            e = RawEvent()
            e.record(st)
        else:
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
        self.events.setdefault(op, [[], []])[which].append(e)

    def totals_ms(self):
        out = {}
        for op, (s, e) in self.events.items():
            out[op] = [a.elapsed_time(b) for a, b in zip(s, e)]
        return out


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def oracle_sample_pass(reps=1):
    """Times the oracle (single-threaded C) on a slice of the embedding table
    planned as its own DBuffer (m=64, 128x128 blocks, E4M3): all five operators.
    Returns (GB/s, elements/s, seconds, description)."""
    import numpy as np
    import oracle
    from workloads import workload
    from workloads.configs import TensorSpec
    w = workload("dense7b")
    emb = w.groups[1].tensors[0]
    spec = TensorSpec("embedding_rows", REF_SAMPLE_ROWS, emb.cols, emb.gran_rows, emb.qblock,
                      emb.quant)
    p = oracle.plan_specs([spec], w.m, None, w.align)
    n = spec.numel
    gen = torch.Generator().manual_seed(0)
    src = (torch.randn(n, generator=gen) * 0.02).numpy()
    grad = np.zeros(p.total, np.float32)
    grad[p.offsets[0]:p.offsets[0] + n] = (torch.randn(n, generator=gen) * 1e-3).numpy()
    acc = np.zeros(p.total, np.float32)
    b16 = np.zeros(p.total, np.uint16)
    dst = np.zeros(n, np.uint16)
    codes = np.zeros(p.total, np.uint8)
    _, ns = oracle.scale_offsets([spec])
    op_bytes = {"pack_cast": 6 * n, "unpack": 4 * n, "scale_accum_zero": 16 * n,
                "norm_nonfinite": 4 * n, "block_quant": 5 * n + 4 * ns}
    nbytes = sum(op_bytes.values())
    op_time = dict.fromkeys(op_bytes, 0.0)
    t0 = time.perf_counter()
    for _ in range(reps):
        for op, fn in (("pack_cast", lambda: oracle.pack(p, [src], b16)),
                       ("unpack", lambda: oracle.unpack(p, b16, [dst])),
                       ("scale_accum_zero", lambda: oracle.scale_accum_zero(p, grad, acc, w.scale)),
                       ("norm_nonfinite", lambda: oracle.norm_nonfinite(p, acc)),
                       ("block_quant", lambda: oracle.block_quant(p, [spec], acc, codes))):
            t1 = time.perf_counter()
            fn()
            op_time[op] += time.perf_counter() - t1
    dt = time.perf_counter() - t0
    desc = (f"{REF_SAMPLE_ROWS}x{emb.cols} slice of the embedding table as one DBuffer "
            f"(m={w.m}, {n} elements), all five operators, x{reps}")
    oracle_sample_pass.last_ops = {op: round(op_bytes[op] * reps / op_time[op] / 1e9, 4)
                                   for op in op_bytes}
    return nbytes * reps / dt / 1e9, n * reps / dt, dt, desc


def _host_cpu():
    """Core count and CPU model of this host (the oracle runs on one core)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    import platform
    return {"nproc": os.cpu_count(), "machine": platform.machine(), "model": model}


def run_reference(args):
    rank, world, local = _dist()
    if rank != 0:
        return 0
    from oracle import build as build_oracle
    build_oracle()
    for _ in range(args.warmup):
        oracle_sample_pass(1)
    t0 = time.perf_counter()
    gbs_l = []
    for _ in range(args.steps):
        gbs, eps, dt, desc = oracle_sample_pass(1)
        gbs_l.append(gbs)
    total = time.perf_counter() - t0
    value = statistics.median(gbs_l)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000 * total / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": _reference_config(),
            "note": ("the oracle's rate per algorithmic byte on a bounded sample of the 7B "
                     "stack; a ratio against the GPU line compares per-byte rates, the "
                     "workloads differ in size"),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": desc,
                             "ops_gbs": getattr(oracle_sample_pass, "last_ops", None),
                             "host": _host_cpu()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _reference_config():
    """The workload the reference arm times: one slice of the dense stack."""
    from workloads import workload
    w = workload("dense7b")
    emb = w.groups[1].tensors[0]
    return {"workload": (f"{REF_SAMPLE_ROWS}x{emb.cols} slice of the 7B-shaped stack's "
                         f"{emb.rows}x{emb.cols} embedding table planned as one DBuffer "
                         f"(m={w.m}, 128x128 E4M3 blocks, s=1/{w.m}): pack_cast, unpack, "
                         "scale_accum_zero, norm_nonfinite, block_quant, once per step"),
            "key": "dense7b_embedding_slice", "elements_per_step": REF_SAMPLE_ROWS * emb.cols,
            "m": w.m, "sample_of": "dense7b"}


def _config_dict(stack, key):
    from workloads import workload
    w = workload(key)
    if key == "dense7b":
        desc = ("7B-shaped dense stack: 32 layers d=4096 ffn=11008 (Wqkv 4096x12288, "
                "Wo 4096x4096, gate/up 4096x11008, down 11008x4096, 2 norms) + embedding "
                "32000x4096; one DBuffer per layer, m=64, 128x128 blocks, E4M3 128x128 "
                "block quant, s=1/64")
    else:
        desc = w.description
    gdt = "bf16" if w.grad_dtype == torch.bfloat16 else "f32"
    quant = sorted({s.quant for g in w.groups for s in g.tensors if s.quant})
    d = {"workload": desc, "key": key,
         "dbuffers": sum(g.repeat for g in w.groups), "m": w.m,
         "ops_per_dbuffer": ["pack_cast f32->bf16", "unpack bf16->bf16",
                             f"scale_accum_zero {gdt} grad", "norm_nonfinite f32",
                             "block_quant " + "+".join(quant) if quant else "block_quant none"],
         "l2": "inputs larger than L2 (129 MB)" if w.total_numel * 4 > 129e6 * 2
               else "inputs near or below L2 size: L2 not flushed (small case)"}
    if stack is not None:
        d["elements_per_step"] = stack.elements
        d["bytes_per_step"] = stack.bytes_per_step
    return d


def _traffic_for(kernel_key, workload_key):
    """dram bytes per launch recorded from an ncu capture (profiles/dram_traffic.txt)
    of this workload, or None if there is none or any source file of that kernel
    changed since (the record carries the files' sha256 prefixes)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    csrc = os.path.join(ROOT, "fsdp_infra_gb300", "csrc")
    with open(path) as f:
        for line in f:
            if line.startswith("#") or "=" not in line:
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if kv.get("op") != kernel_key:
                continue
            if kv.get("workload", "").split("-")[0] != workload_key:
                continue
            for name, sha in zip(kv["files"].split(","), kv["sha"].split(",")):
                try:
                    with open(os.path.join(csrc, name), "rb") as fh:
                        if hashlib.sha256(fh.read()).hexdigest()[:16] != sha:
                            return None
                except OSError:
                    return None
            return float(kv["bytes_per_launch"])
    return None


def op_alone_ms(stack, op, eager, passes=3, min_launches=32):
    """Milliseconds of one pass of `op` over every DBuffer: the launches back to
    back (captured as one graph unless eager), one untimed pass, then `passes`
    timed ones between two events.  Each pass moves far more than L2 holds.  A
    workload of few DBuffers repeats its pass inside the graph until it holds at
    least `min_launches` DBuffer launches, so that the graph's own launch cost is
    not charged to one or two kernels."""
    reps = max(1, -(-min_launches // max(1, len(stack.dbufs))))

    def one():
        for _ in range(reps):
            stack.run_op(op)

    graph = None
    if not eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one()
    run = graph.replay if graph is not None else one
    run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(passes):
        run()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / (passes * reps)


def step_alone_ms(stack, eager, passes=3, min_steps=32):
    """Milliseconds of one whole step (every operator over every DBuffer), timed
    like op_alone_ms: a workload of few DBuffers repeats its step inside one
    graph until it holds at least `min_steps` DBuffer steps."""
    reps = max(1, -(-min_steps // max(1, len(stack.dbufs))))

    def one():
        for _ in range(reps):
            stack.step()

    graph = None
    if not eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one()
    run = graph.replay if graph is not None else one
    run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(passes):
        run()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / (passes * reps)


PER_CONFIG = ("tiny", "llama_layer", "moe", "mixed")
L2_BYTES = 129e6


def l2_label(numel):
    """How a workload's buffers sit against the 129 MB L2 (launches back to back,
    no flush between them)."""
    f32 = numel * 4
    if f32 > 2 * L2_BYTES:
        return "buffers larger than L2 (129 MB)"
    if f32 > L2_BYTES:
        return (f"fp32 buffers ({f32 / 1e6:.0f} MB) larger than L2 (129 MB), bf16 buffer "
                f"({f32 / 2e6:.0f} MB) smaller: partly L2-resident between launches")
    return "small case: L2-resident and launch-bound, not an HBM rate"


def run_per_config(args, device, peak):
    """The other four workloads, each planned and stepped alone on this GPU
    (outside the timed region of the headline step): per operator its launches
    back to back in one graph (at least 32 launches, 3 passes), and the whole
    step the same way.  GB/s = algorithmic bytes (tensor ranges only) / time;
    elements/s = the workload's elements / time."""
    from workloads import workload
    out = {}
    for key in PER_CONFIG:
        w = workload(key)
        st = Stack(w, device)
        torch.cuda.synchronize()
        for _ in range(max(args.warmup, 1)):
            st.step()
        torch.cuda.synchronize()
        ops = {}
        for op in ("pack_cast", "unpack", "scale_accum_zero", "norm_nonfinite", "block_quant"):
            if st.op_bytes.get(op, 0) == 0:
                continue
            ms = op_alone_ms(st, op, args.eager)
            gbs = st.op_bytes[op] / (ms / 1e3) / 1e9
            ops[op] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                       "elements_per_s": round(st.elements / (ms / 1e3), 1)}
        ms = step_alone_ms(st, args.eager)
        gbs = st.bytes_per_step / (ms / 1e3) / 1e9
        out[key] = {"workload": w.description, "m": w.m, "dbuffers": len(st.dbufs),
                    "elements": st.elements, "bytes_per_step": st.bytes_per_step,
                    "grad_dtype": "bf16" if w.grad_dtype == torch.bfloat16 else "f32",
                    "l2": l2_label(w.total_numel),
                    "step": {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                             "elements_per_s": round(st.elements / (ms / 1e3), 1)},
                    "ops": ops}
        for d in st.dbufs:
            d["kind"]["db"].close()
        del st
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    from fsdp_infra_gb300 import build as _b  # noqa: F401  (library must already be built)
    from workloads import workload
    w = workload(args.workload)
    stack = Stack(w, device)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(args.warmup, 0)):
        stack.step()
    torch.cuda.synchronize()
    peak, peak_kind = _peaks()

    # Per-operator breakdown (outside the timed region): one step with timing
    # events around every operator, captured as a graph so that host-side work
    # between launches does not show up as GPU time (eager with --eager).
    probe = OpTimers(raw=not args.eager)
    if args.eager:
        stack.step(probe)
    else:
        probe_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(probe_graph):
            stack.step(probe)
        probe_graph.replay()
    torch.cuda.synchronize()
    per_op_eager = probe.totals_ms()
    # Each operator alone: its launches over every DBuffer back to back (as in the
    # step, without events between them), timed over a few passes; the figures
    # with events around every launch stay beside them.
    ops = {}
    for op, durs in per_op_eager.items():
        if stack.op_bytes.get(op, 0) == 0 or sum(durs) <= 0:
            continue
        ms = op_alone_ms(stack, op, args.eager)
        ops[op] = {"ms_per_step": round(ms, 4),
                   "gbs": round(stack.op_bytes[op] / (ms / 1e3) / 1e9, 1),
                   "frac": round(stack.op_bytes[op] / (ms / 1e3) / 1e9 / peak, 4),
                   "evented_ms_per_step": round(sum(durs), 4),
                   "evented_mean_launch_ms": round(statistics.mean(durs), 4)}
    dom = max((k for k in per_op_eager if stack.op_bytes.get(k, 0) > 0),
              key=lambda k: sum(per_op_eager[k]))

    # Timed region: K steps; by default captured once as a CUDA graph (all
    # launches of the K steps) and replayed once untimed, then once timed.
    # Timing events bracket each launch of the dominant operator in the middle
    # step only: an event node between two kernels breaks their programmatic
    # launch edge, and events around that operator's launches in every step cost
    # about 1% of the step time.
    timers = OpTimers(only=dom, raw=not args.eager)
    timed_step = args.steps // 2
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                stack.step(timers if i == timed_step else None)
        graph.replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(device)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            stack.step(timers if i == timed_step else None)
    t_end.record()
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), device)
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(stack.bytes_per_step, ms_per_step, world)
    per_op = timers.totals_ms()

    # achieved for the dominant operator: algorithmic bytes of one launch on a
    # DBuffer of the group that carries most of the elements (the 32 layers of
    # the dense stack) over the mean duration of those launches in the middle timed step.
    big = max(range(len(stack.w.groups)),
              key=lambda gi: stack.w.groups[gi].numel * stack.w.groups[gi].repeat)
    g0 = stack.w.groups[big]
    big_db = next(d["kind"]["db"] for d in stack.dbufs if d["kind"]["gi"] == big)
    if dom == "block_quant":
        layer_bytes = 5 * sum(s.numel for s in g0.tensors if s.quant) + 4 * big_db.n_scales
    else:
        layer_bytes = stack.per_elem[dom] * g0.numel
    kinds = [d["kind"]["gi"] for d in stack.dbufs]
    layer_durs = [d for i, d in enumerate(per_op[dom]) if kinds[i % len(kinds)] == big]
    mean_layer_ms = statistics.mean(layer_durs)
    achieved = layer_bytes / (mean_layer_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "bytes_per_launch": layer_bytes,
                "traffic": _traffic_for(dom, stack.w.key)}

    # ---- the next row: fused AdamW step over every DBuffer (separate timing)
    adamw = None if args.no_adamw else run_adamw(stack, args, world, peak, barrier)
    adamw8 = None if args.no_adamw else run_adamw8(stack, args, world, peak, barrier)
    adamw8_128 = (None if args.no_adamw else
                  run_adamw8(stack, args, world, peak, barrier, block=(128, 128)))
    gather = None if args.no_adamw else run_gather(stack, args, world, peak, barrier)

    # ---- end to end: host inputs (pinned) -> device, operators, results -> host
    e2e = None if args.no_e2e else run_e2e(stack, args, world)

    # ---- the other workloads, each alone (not part of the timed step)
    per_config = None
    if not args.no_per_config and args.workload == "dense7b":
        per_config = run_per_config(args, device, peak)

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            import oracle
            oracle.build()
            gbs, eps, dt, desc = oracle_sample_pass(1)
            cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": desc, "seconds": round(dt, 2),
                   "note": "per-byte rate on a bounded sample, not the whole step",
                   "ops_gbs": getattr(oracle_sample_pass, "last_ops", None),
                   "host": _host_cpu()}
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": _config_dict(stack, args.workload),
                "params_per_s": round(world * stack.elements / (ms_per_step / 1e3), 1),
                "frac_of_peak": round(value / world / peak, 4), "peak_kind": peak_kind,
                "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": stack.launches_per_step * args.steps,
                "next_rows": ({"adamw": adamw, "adamw8": adamw8, "adamw8_128x128": adamw8_128,
                               "gather_scatter": gather} if adamw else None),
                "launch": "eager" if args.eager else "cuda_graph (K steps captured once, replayed)",
                "ops_note": ("per operator, outside the timed region: its launches over every "
                             "DBuffer back to back, timed over 3 passes" +
                             ("" if args.eager else " of one graph") +
                             (f" (each pass repeated {-(-32 // len(stack.dbufs))}x, "
                              "at least 32 launches)" if len(stack.dbufs) < 32 else "") +
                             "; evented_*: one step with events around every launch"),
                "clocks": clock_info, "ops": ops, "per_config": per_config,
                "per_config_note": ("each workload planned and stepped alone after the timed "
                                    "region: per operator its launches back to back in one "
                                    "graph (at least 32 launches, 3 passes); step = all five "
                                    "operators, timed the same way; frac of the measured "
                                    "copy peak")}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _exchange_config(key, world):
    """The workload's config with its DBuffers re-planned for `world` ranks."""
    cfg = _config_dict(None, key)
    desc = re.sub(r"\bm=\d+", f"m={world}", cfg["workload"])
    desc = re.sub(r"\bs=1/\d+", f"s=1/{world}", desc)
    cfg["workload"] = desc + "; every group re-planned evenly over the ranks for the exchange"
    return dict(cfg, m=world, parallelism=f"fsdp{world} (one shard slice per rank)")


def run_exchange(args):
    """--exchange: the data-parallel step with its collectives, one rank per GPU
    (fsdp_infra_gb300.exchange.ShardedStep).  Every DBuffer of the workload is
    re-planned with m = world size (an even plan, one slice per rank); a step runs,
    for every DBuffer, copy-in of the rank's gradients, ReduceScatter, the slice's
    scale/accumulate/zero, sharded norm (AllReduce of the partial sums and the
    flag) and block quantisation, then the cast of the rank's master pieces,
    AllGather and copy-out.  Launched eagerly; the step time includes the
    collectives.  `value` counts the group operators' algorithmic bytes of every
    rank (full-buffer pack and unpack, slice sac, norm and quantisation);
    `collective_bytes_per_rank` the bytes each rank sends into the collectives.
    With one GPU the process group has one rank and the collectives copy."""
    import torch.distributed as dist
    from fsdp_infra_gb300 import DBuffer
    from fsdp_infra_gb300.exchange import ShardedStep
    from workloads import workload, param_values
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    else:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1, device_id=device)
    w = workload(args.workload)
    peak, peak_kind = _peaks()
    kinds, items = [], []
    for gi, g in enumerate(w.groups):
        full = DBuffer(g.tensors, world, None, w.align, device=device).upload()
        loc = full.slice(rank).upload()
        k = {"full": full, "local": loc, "step": ShardedStep(full, loc, rank, world),
             "grad_full": torch.zeros(full.total, dtype=torch.float32, device=device),
             "grad_local": torch.zeros(loc.total, dtype=torch.float32, device=device),
             "acc_local": torch.zeros(loc.total, dtype=torch.float32, device=device),
             "buf_local": torch.zeros(loc.total, dtype=torch.bfloat16, device=device),
             "buf_full": torch.zeros(full.total, dtype=torch.bfloat16, device=device),
             "codes": torch.zeros(max(loc.total, 1), dtype=torch.uint8, device=device),
             "scales": torch.zeros(max(loc.n_scales, 1), dtype=torch.float32, device=device)}
        kinds.append(k)
        for r in range(g.repeat):
            master = [param_values(w, gi, t, device=device, seed=1000 * r + gi)
                      for t in range(len(g.tensors))]
            gen = torch.Generator(device=device)
            gen.manual_seed(4321 + 97 * rank + r)
            grads = [torch.randn(s.rows, s.cols, generator=gen, device=device).mul_(w.grad_std)
                     for s in g.tensors]
            compute = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=device)
                       for s in g.tensors]
            for x in (master, grads, compute):
                full.ptr_table(x)
            items.append((k, master, grads, compute))

    def step():
        for k, master, grads, compute in items:
            k["step"].reduce_gradients(grads, k["grad_full"], k["grad_local"], k["acc_local"],
                                       1.0 / world, codes=k["codes"], scales=k["scales"])
            k["step"].gather_parameters(master, k["buf_local"], k["buf_full"], compute)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    clocks = ClockSampler(device)
    clocks.start()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        step()
    e.record()
    torch.cuda.synchronize()
    dist.barrier()
    clock_info = clocks.stop()
    ms = max_over_ranks(s.elapsed_time(e), device) / args.steps
    op_bytes, coll = 0, 0
    for k, master, grads, compute in items:
        full, loc = k["full"], k["local"]
        E = sum(full.numel)
        qe = sum(n for n, sp in zip(loc.piece_numels, full.specs) if sp.quant)
        el = sum(loc.piece_numels)
        op_bytes += 8 * E + 4 * E          # copy-in fp32 -> fp32, copy-out bf16 -> bf16
        op_bytes += 16 * el + 4 * el + 6 * el + 5 * qe + 4 * loc.n_scales  # sac, norm, cast, quant
        coll += 4 * full.total + 2 * loc.total + 16 * full.n
    value = world * op_bytes / (ms / 1e3) / 1e9
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
                "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic", "mode": "exchange",
                "config": _exchange_config(args.workload, world),
                "collective_bytes_per_rank": coll, "op_bytes_per_rank": op_bytes,
                "frac_of_peak": round(value / world / peak, 4), "peak_kind": peak_kind,
                "launch": "eager, collectives on the default stream", "clocks": clock_info}
        print(json.dumps(line), flush=True)
    for k in kinds:
        k["local"].close()
        k["full"].close()
    dist.destroy_process_group()
    return 0


def run_adamw(stack, args, world, peak, barrier):
    """The fused AdamW step (dbuf_adamw_step) over every DBuffer of the workload:
    fp32 master parameters, the accumulated gradients and both moments in the
    plan's layout, clipped to max_norm 1.0 with each DBuffer's own device norm and
    non-finite flag from the step.  K steps captured once as a CUDA graph and
    timed as one replay; 28 algorithmic bytes per element (read p, g, m, v; write
    p, m, v)."""
    device = stack.device
    for d in stack.dbufs:
        k = d["kind"]
        if "p32" not in k:
            k["p32"] = torch.zeros_like(k["acc"])
            k["m32"] = torch.zeros_like(k["acc"])
            k["v32"] = torch.zeros_like(k["acc"])
            db = k["db"]
            for t, x in enumerate(d["params"]):
                k["p32"][db.offsets[t]:db.offsets[t] + x.numel()].copy_(x.reshape(-1))

    def step(i):
        for d in stack.dbufs:
            k = d["kind"]
            k["db"].adamw_step(k["p32"], k["acc"], k["m32"], k["v32"], step=i, lr=1e-4,
                               betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, max_norm=1.0,
                               total_norm=d["out"][1], nonfinite=d["out"][2])

    for i in range(1, max(args.warmup, 1) + 1):
        step(i)
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(10 + i)
        graph.replay()
        torch.cuda.synchronize()
    barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(10 + i)
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), device) / args.steps
    nbytes = 28 * stack.elements
    gbs = job_throughput(nbytes, ms, world)
    return {"op": "dbuf_adamw_step (fp32 params/grads/moments, clip to the step's device norm)",
            "gbs": round(gbs, 1), "ms_per_step": round(ms, 4),
            "params_per_s": round(world * stack.elements / (ms / 1e3), 1),
            "frac_of_peak": round(gbs / world / peak, 4), "bytes_per_elem": 28,
            "launches_per_step": len(stack.dbufs),
            "traffic_layer_launch": _traffic_for("adamw", stack.w.key),
            "algorithmic_layer_launch": 28 * stack.w.groups[0].numel}


def run_adamw8(stack, args, world, peak, barrier, block=(32, 32)):
    """8-bit AdamW (dbuf_adamw8_step) over every DBuffer of the workload, each
    group re-planned as the 8-bit Adam experiment shards it (block x block INT8
    blocks at block-row granularity for matrices; 32x32 in the experiment,
    128x128 the big-block kernel's case): fp32 master parameters and gradients,
    8-bit block moments, compact fp32 moments for vectors; clipped to max_norm
    1.0 with the group's device norm.  One plan and one set of buffers per group
    kind, stepped once per DBuffer (the buffers exceed L2).  K steps captured
    once as a CUDA graph and timed as one replay.  Algorithmic bytes: 16 per
    element of a quantised tensor (read p, g and two codes; write p and two
    codes), 28 per element of the others, 16 per block (two scales read and
    written)."""
    from fsdp_infra_gb300 import DBuffer
    from workloads import grad_values, param_values
    from workloads.configs import adam8_group
    device = stack.device
    w = stack.w
    kinds = {}
    for gi, g in enumerate(w.groups):
        g8 = adam8_group(g, block)
        db = DBuffer(g8.tensors, w.m, None, w.align, device=device).upload()
        p32 = torch.zeros(db.total, dtype=torch.float32, device=device)
        g32 = torch.zeros(db.total, dtype=torch.float32, device=device)
        for t, spec in enumerate(g8.tensors):
            o = db.offsets[t]
            p32[o:o + spec.numel].copy_(param_values(w, gi, t, device=device).reshape(-1))
            g32[o:o + spec.numel].copy_(grad_values(w, gi, t, device=device).reshape(-1).float())
        out = db.norm_nonfinite(g32)
        qe = sum(spec.numel for spec in g8.tensors if spec.quant)
        pe = sum(spec.numel for spec in g8.tensors if not spec.quant)
        # launches: the pipelined kernel (the stage kernel, or the big-block kernel
        # for blocks of two stages) once per 16 quantised tensors (the tensor maps
        # one launch carries), the register kernel once for the rest
        nq = sum(1 for spec in g8.tensors if spec.quant and spec.numel)
        rest = any(spec.numel and not spec.quant for spec in g8.tensors)
        kinds[gi] = {"db": db, "p": p32, "g": g32, "state": db.new_adamw8_state(), "out": out,
                     "bytes": 16 * qe + 28 * pe + 16 * db.n_scales,
                     "launches": (nq + 15) // 16 + (1 if rest else 0)}
    order = [d["kind"]["gi"] for d in stack.dbufs]

    def step(i):
        for gi in order:
            k = kinds[gi]
            k["db"].adamw8_step(k["p"], k["g"], k["state"], step=i, lr=1e-4, betas=(0.9, 0.95),
                                eps=1e-8, weight_decay=0.1, max_norm=1.0, total_norm=k["out"][1],
                                nonfinite=k["out"][2])

    for i in range(1, max(args.warmup, 1) + 1):
        step(i)
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(10 + i)
        graph.replay()
        torch.cuda.synchronize()
    barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(10 + i)
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), device) / args.steps
    nbytes = sum(kinds[gi]["bytes"] for gi in order)
    gbs = job_throughput(nbytes, ms, world)
    elems = sum(kinds[gi]["db"].total for gi in order)
    blk = sorted({spec.qblock for g in w.groups for spec in adam8_group(g, block).tensors
                  if spec.quant})
    return {"op": "dbuf_adamw8_step (fp32 params/grads, 8-bit block moments, clip to the "
                  "group's device norm)",
            "blocks": [list(b) for b in blk], "gbs": round(gbs, 1), "ms_per_step": round(ms, 4),
            "params_per_s": round(world * stack.elements / (ms / 1e3), 1),
            "frac_of_peak": round(gbs / world / peak, 4),
            "bytes_per_step": nbytes, "flat_elements_per_step": elems,
            "launches_per_step": sum(kinds[gi]["launches"] for gi in order),
            "traffic_layer_launch": _traffic_for("adamw8", stack.w.key),
            "algorithmic_layer_launch": kinds[0]["bytes"]}


def run_gather(stack, args, world, peak, barrier):
    """Whole-matrix gather and scatter (dbuf_gather + dbuf_scatter) of every
    tensor of every DBuffer: the m shards are the slices [B_k, B_{k+1}) of the
    group's fp32 accumulator, the matrices separate fp32 buffers.  One gather
    and one scatter per DBuffer per step; K steps captured once as a CUDA graph
    and timed as one replay.  Algorithmic bytes: 16 per element (each copy
    reads and writes 4)."""
    device = stack.device
    for d in stack.dbufs:
        k = d["kind"]
        if "mats" not in k:
            db = k["db"]
            b = db.shard_bounds
            k["shards"] = [k["acc"][b[i]:b[i + 1]] for i in range(db.m)]
            k["mats"] = [torch.empty(s.numel, dtype=torch.float32, device=device)
                         for s in k["spec"].tensors]

    def step():
        for d in stack.dbufs:
            k = d["kind"]
            k["db"].gather(k["shards"], k["mats"])
            k["db"].scatter(k["mats"], k["shards"])

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                step()
        graph.replay()
        torch.cuda.synchronize()
    barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    if graph is not None:
        graph.replay()
    else:
        for _ in range(args.steps):
            step()
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), device) / args.steps
    nbytes = 16 * stack.elements
    gbs = job_throughput(nbytes, ms, world)
    return {"op": "dbuf_gather + dbuf_scatter (every tensor, fp32, m shard slices)",
            "gbs": round(gbs, 1), "ms_per_step": round(ms, 4),
            "frac_of_peak": round(gbs / world / peak, 4), "bytes_per_elem": 16,
            "launches_per_step": 2 * len(stack.dbufs),
            "traffic_layer_launch": {"gather": _traffic_for("gather", stack.w.key),
                                     "scatter": _traffic_for("scatter", stack.w.key)},
            "algorithmic_layer_launch": 8 * stack.w.groups[0].numel}


def run_e2e(stack, args, world):
    """Same step through the public API, with this step's inputs copied from
    pinned host memory (fp32 master params and fp32 gradients of every DBuffer)
    and the results (norms, non-finite flags) read back to the host.  The copies
    run on a side stream and overlap the operators of the previous DBuffer: each
    DBuffer kind has two gradient buffers used alternately, and events order
    every reuse (a parameter tensor is refilled only after the previous step's
    pack read it; a gradient buffer only after the sac that read it)."""
    device = stack.device
    host = {}
    for d in stack.dbufs:
        k = d["kind"]
        if id(k) in host:
            continue
        g = k["spec"]
        db = k["db"]
        hp = [torch.empty(s.numel, dtype=torch.float32, pin_memory=True) for s in g.tensors]
        hg = [torch.empty(s.numel, dtype=stack.w.grad_dtype, pin_memory=True) for s in g.tensors]
        for t, s in enumerate(g.tensors):
            hp[t].copy_(d["params"][t].reshape(-1))
            hg[t].copy_(k["grad"][db.offsets[t]:db.offsets[t] + s.numel])
        if "grad2" not in k:
            k["grad2"] = torch.zeros_like(k["grad"])
        host[id(k)] = (hp, hg, torch.empty(len(g.tensors) + 2, dtype=torch.float32,
                                           pin_memory=True))
    h2d = 0
    d2h = 0
    for d in stack.dbufs:
        hp, hg, _ = host[id(d["kind"])]
        h2d += sum(x.numel() * x.element_size() for x in hp) + sum(x.numel() * x.element_size() for x in hg)
        d2h += (len(hp) + 2) * 4

    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    nd = len(stack.dbufs)
    pack_done = [None] * nd           # per DBuffer: its params were read
    grad_free = {}                    # (kind id, slot) -> event: that gradient buffer was read
    use = {}                          # kind id -> running count (slot = count % 2)

    def step():
        for i, d in enumerate(stack.dbufs):
            k, db = d["kind"], d["kind"]["db"]
            hp, hg, hout = host[id(k)]
            n = use.get(id(k), 0)
            use[id(k)] = n + 1
            slot = n % 2
            grad = k["grad"] if slot == 0 else k["grad2"]
            with torch.cuda.stream(copy):
                if pack_done[i] is not None:
                    copy.wait_event(pack_done[i])
                if (id(k), slot) in grad_free:
                    copy.wait_event(grad_free[(id(k), slot)])
                for t in range(len(hp)):
                    d["params"][t].view(-1).copy_(hp[t], non_blocking=True)
                    o = db.offsets[t]
                    grad[o:o + hg[t].numel()].copy_(hg[t], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(copy)
            compute.wait_event(ready)
            db.pack_cast(d["params"], k["buf16"], stream=compute)
            ev = torch.cuda.Event()
            ev.record(compute)
            pack_done[i] = ev
            db.unpack(k["buf16"], d["compute"], stream=compute)
            db.scale_accum_zero(grad, k["acc"], stack.w.scale, stream=compute)
            ev = torch.cuda.Event()
            ev.record(compute)
            grad_free[(id(k), slot)] = ev
            norms, tot, flag = db.norm_nonfinite(k["acc"], out=d["out"], stream=compute)
            db.block_quant(k["acc"], codes=k["codes"], scales=k["scales"], stream=compute)
            n_t = len(hp)
            hout[:n_t].copy_(norms, non_blocking=True)
            hout[n_t:n_t + 1].copy_(tot, non_blocking=True)
            hout[n_t + 1:n_t + 2].copy_(flag.view(torch.float32), non_blocking=True)
        compute.synchronize()

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    steps = max(1, min(args.steps, 5))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, device)
    value = job_throughput(stack.bytes_per_step, 1e3 * dt / steps, world)
    return {"value": round(value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1000 * dt / steps, 3),
            "h2d_gbs": round(h2d * steps / dt / 1e9, 1),
            "note": "host->device copies on a side stream overlap the operators; "
                    "timed with the host clock around whole steps"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adamw", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--exchange", action="store_true",
                    help="the sharded step with its collectives (m = number of GPUs) instead "
                         "of independent replicas of the group-operator pass")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one instead of as one CUDA graph")
    ap.add_argument("--workload", default="dense7b",
                    choices=["dense7b", "llama_layer", "tiny", "moe", "mixed"],
                    help="dense7b is the benchmark; the others are small or alternate "
                         "cases (profiling captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.exchange:
        return run_exchange(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
