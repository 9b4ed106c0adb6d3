"""The five synthetic tensor-group workloads and their seeded value generators.

Shapes follow the model families that the veScale-FSDP and PyTorch FSDP pages
train on (transformer layers, a 7B-shaped dense stack, an MoE expert group, and a
Muon/Shampoo-style mixed group of many small tensors).  No dataset and no trained
weights are involved: every value is drawn from a seeded normal distribution.

A tensor is row-major ``[rows, cols]``; a 1-D vector is ``[n, 1]``.  ``gran_rows``
is the RaggedShard sharding granularity in rows (a shard boundary may fall inside
the tensor only at a multiple of ``gran_rows`` rows from its start); 0 means the
whole tensor is one indivisible unit.  ``qblock`` is the quantisation block
``(rows, cols)`` and ``quant`` its code format (None, ``"e4m3"`` or ``"int8"``).
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch


@dataclass(frozen=True)
class TensorSpec:
    name: str
    rows: int
    cols: int
    gran_rows: int          # 0 = whole tensor is one unit
    qblock: Tuple[int, int] = (0, 0)
    quant: Optional[str] = None   # None | "e4m3" | "int8"
    kind: str = "matrix"    # "matrix" | "norm" | "vector"

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class GroupSpec:
    """One DBuffer: an ordered tensor group planned into one flat buffer."""
    name: str
    tensors: Tuple[TensorSpec, ...]
    repeat: int = 1         # identical groups (e.g. 32 transformer layers)

    @property
    def numel(self) -> int:
        return sum(t.numel for t in self.tensors)


@dataclass(frozen=True)
class Workload:
    key: str
    description: str
    groups: Tuple[GroupSpec, ...]
    m: int                              # number of shard slices
    local_units: Optional[Tuple[int, ...]]  # None = even shards
    align: int                          # alignment in elements of S and of every offset
    grad_dtype: torch.dtype             # dtype of the gradient buffer
    param_std: float = 0.02
    grad_std: float = 1e-3
    accum_steps: int = 1
    seed: int = 0
    notes: str = ""

    @property
    def scale(self) -> float:
        """Gradient scale s = 1/m (mean over the m data-parallel slices)."""
        return 1.0 / self.m

    @property
    def total_numel(self) -> int:
        return sum(g.numel * g.repeat for g in self.groups)


ALIGN = 16


def _mat(name, r, c, gran, qb=(0, 0), quant=None):
    return TensorSpec(name, r, c, gran, qb, quant, "matrix")


def _norm(name, n):
    return TensorSpec(name, n, 1, 1, (0, 0), None, "norm")


def _tiny_transformer() -> Workload:
    d, f = 256, 1024
    ts: List[TensorSpec] = []
    for layer in range(2):
        q = dict(gran=128, qb=(128, 128), quant="e4m3")
        for w in ("wq", "wk", "wv", "wo"):
            ts.append(_mat(f"l{layer}.{w}", d, d, **q))
        ts.append(_mat(f"l{layer}.w1", d, f, **q))
        ts.append(_mat(f"l{layer}.w2", f, d, **q))
        ts.append(_norm(f"l{layer}.attn_norm", d))
        ts.append(_norm(f"l{layer}.ffn_norm", d))
    g = GroupSpec("tiny2layer", tuple(ts))
    return Workload(
        key="tiny",
        description="tiny 2-layer transformer group d=256 ffn=1024, 16 tensors, m=4, "
                    "128x128 blocks, E4M3 128x128 quant",
        groups=(g,), m=4, local_units=None, align=ALIGN, grad_dtype=torch.float32)


def _llama_layer() -> Workload:
    d, f = 2048, 5632
    q = dict(gran=128, qb=(128, 128), quant="e4m3")
    ts = (
        _mat("wqkv", d, 3 * d, **q),
        _mat("wo", d, d, **q),
        _mat("w_gate", d, f, **q),
        _mat("w_up", d, f, **q),
        _mat("w_down", f, d, **q),
        _norm("attn_norm", d),
        _norm("ffn_norm", d),
    )
    return Workload(
        key="llama_layer",
        description="one Llama-style layer d=2048 ffn=5632, m=8, 128x128 blocks, "
                    "E4M3 128x128 quant, 4-step grad accumulation",
        groups=(GroupSpec("layer", ts),), m=8, local_units=None, align=ALIGN,
        grad_dtype=torch.float32, accum_steps=4,
        notes="one +inf injected into the gradients of 1 of 10 runs")


def _dense7b() -> Workload:
    d, f, vocab = 4096, 11008, 32000
    q = dict(gran=128, qb=(128, 128), quant="e4m3")
    layer = (
        _mat("wqkv", d, 3 * d, **q),
        _mat("wo", d, d, **q),
        _mat("w_gate", d, f, **q),
        _mat("w_up", d, f, **q),
        _mat("w_down", f, d, **q),
        _norm("attn_norm", d),
        _norm("ffn_norm", d),
    )
    emb = (_mat("embedding", vocab, d, **q),)
    return Workload(
        key="dense7b",
        description="7B-shaped dense stack: 32 layers d=4096 ffn=11008 + embedding "
                    "32000x4096, one DBuffer per layer, m=64, 128x128 blocks, "
                    "E4M3 128x128 quant, s=1/64",
        groups=(GroupSpec("layer", layer, repeat=32), GroupSpec("embedding", emb)),
        m=64, local_units=None, align=ALIGN, grad_dtype=torch.float32)


def _moe_group(seed: int = 0) -> Workload:
    d, fe, experts, m = 2048, 1408, 64, 16
    ts: List[TensorSpec] = []
    for e in range(experts):
        q = dict(gran=1, qb=(1, 128), quant="int8")
        ts.append(_mat(f"e{e}.gate", d, fe, **q))
        ts.append(_mat(f"e{e}.up", d, fe, **q))
        ts.append(_mat(f"e{e}.down", fe, d, **q))
    ts.append(_mat("router", d, experts, gran=1, qb=(1, 128), quant="int8"))
    rng = random.Random(seed)
    units = tuple(rng.randint(1, 4) for _ in range(m))
    return Workload(
        key="moe",
        description="MoE layer group: 64 experts gate/up 2048x1408 down 1408x2048 + "
                    "router 2048x64, row-wise RaggedShard with uneven local_units "
                    "U{1..4}, m=16, bf16 grads, INT8 1x128 quant",
        groups=(GroupSpec("moe", tuple(ts)),), m=m, local_units=units, align=ALIGN,
        grad_dtype=torch.bfloat16, seed=seed)


def _mixed_group(seed: int = 0, count: int = 2000) -> Workload:
    rng = random.Random(seed)
    hi = math.log(4 * 1024 * 1024)
    ts: List[TensorSpec] = []
    for i in range(count):
        n = int(round(math.exp(rng.uniform(0.0, hi))))
        n = max(n, 1)
        if n >= 4096:
            r = 64 * max(1, int(round(math.sqrt(n) / 64)))
            c = 64 * max(1, int(round(n / r / 64)))
            ts.append(_mat(f"m{i}", r, c, gran=0))
        else:
            ts.append(TensorSpec(f"v{i}", n, 1, 1, (0, 0), None, "vector"))
    return Workload(
        key="mixed",
        description="Muon/Shampoo-style mixed group: 2000 tensors, sizes log-uniform "
                    "1..4M elements, whole-matrix blocks for matrices, element "
                    "granularity for vectors, m=32",
        groups=(GroupSpec("mixed", tuple(ts)),), m=32, local_units=None, align=ALIGN,
        grad_dtype=torch.float32, seed=seed)


def adam8_group(group: GroupSpec, block=(32, 32)) -> GroupSpec:
    """The group as the 8-bit Adam experiment shards it: every matrix with
    block x block INT8 quantisation blocks and block[0]-row sharding
    granularity; other tensors unchanged."""
    ts = tuple(TensorSpec(t.name, t.rows, t.cols, block[0], tuple(block), "int8", t.kind)
               if t.kind == "matrix" else t for t in group.tensors)
    return GroupSpec(group.name + "_adam8", ts, group.repeat)


WORKLOADS = {
    "tiny": _tiny_transformer,
    "llama_layer": _llama_layer,
    "dense7b": _dense7b,
    "moe": _moe_group,
    "mixed": _mixed_group,
}


def workload(key: str) -> Workload:
    return WORKLOADS[key]()


def _tensor_seed(seed: int, group_index: int, tensor_index: int, stream: int) -> int:
    return (((seed * 1000003 + group_index) * 1000003 + tensor_index) * 7 + stream) % (2 ** 63)


def param_values(w: Workload, group_index: int, tensor_index: int,
                 device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    """fp32 parameter values of one tensor: N(0, param_std); norm weights are 1.0."""
    spec = w.groups[group_index].tensors[tensor_index]
    if spec.kind == "norm":
        return torch.ones(spec.rows, spec.cols, dtype=torch.float32, device=device)
    s = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(_tensor_seed(s, group_index, tensor_index, 1))
    x = torch.randn(spec.rows, spec.cols, generator=gen, dtype=torch.float32, device=device)
    return x.mul_(w.param_std)


def grad_values(w: Workload, group_index: int, tensor_index: int, device="cpu",
                seed: Optional[int] = None, step: int = 0) -> torch.Tensor:
    """Gradient values of one tensor in the workload's grad dtype: N(0, grad_std)."""
    spec = w.groups[group_index].tensors[tensor_index]
    s = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(_tensor_seed(s, group_index, tensor_index, 2 + 2 * step))
    x = torch.randn(spec.rows, spec.cols, generator=gen, dtype=torch.float32, device=device)
    return x.mul_(w.grad_std).to(w.grad_dtype)


def inf_injection(w: Workload, runs: int = 10, seed: int = 0):
    """(run, tensor index, element index) of the single +inf injected into 1 of `runs`
    gradient runs (group 0)."""
    rng = random.Random(seed + 12345)
    r = rng.randrange(runs)
    ts = w.groups[0].tensors
    t = rng.randrange(len(ts))
    i = rng.randrange(ts[t].numel)
    return r, t, i


def random_tiny_group(rng: random.Random, max_tensors: int = 5, max_rows: int = 8,
                      max_cols: int = 4) -> List[TensorSpec]:
    """A small random tensor group for exhaustive and randomized layout checks."""
    n = rng.randint(1, max_tensors)
    out = []
    for i in range(n):
        r = rng.randint(0, max_rows) if rng.random() < 0.05 else rng.randint(1, max_rows)
        c = rng.randint(1, max_cols)
        gran = rng.choice([0, 1, 1, 2, 3, 4, r if r > 0 else 1])
        out.append(TensorSpec(f"t{i}", r, c, gran))
    return out
