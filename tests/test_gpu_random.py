"""Seeded random groups against the oracle.

Each case draws a tensor group (vectors and matrices of random sizes, empty
tensors, block shapes 128x128, 64x128, 32x32, 16x16, 1x128, 1x64 and an odd 5x4
with ragged edges, E4M3 and INT8, unquantised matrices at 1-, 4- and
whole-tensor row granularity), a shard count m in 1..9, even or uneven
local_units, alignment 1 or 16, and fp32 or bf16 gradients; every operator runs
on the GPU and is compared with the oracle on whole buffers (two accumulation
steps).  The 8-bit AdamW cases draw groups the same way and take two steps
against the oracle.  The cases are reproducible from their seed; the
DBUF_RANDOM_CASES environment variable runs more seeds of both.  Larger groups
(20-70 tensors of up to a few million elements, 128x96, 64x256 and 256x64
blocks too) take every step operator and two 8-bit AdamW steps
(DBUF_LARGE_RANDOM seeds, two by default).
"""
import os

import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec

from test_gpu_optim8 import Case
from test_gpu_parity import full_group_parity

pytestmark = pytest.mark.gpu

BLOCKS = [(128, 128), (64, 128), (32, 32), (16, 16), (1, 128), (1, 64), (5, 4)]
# DBUF_RANDOM_CASES=N widens both sweeps to N seeds (a longer soak of the same draws)
_N = int(os.environ.get("DBUF_RANDOM_CASES", "0"))
N_GROUPS, N_ADAMW8 = (_N, _N) if _N > 0 else (24, 10)


def random_group(rng):
    specs = []
    for t in range(int(rng.integers(1, 13))):
        kind = rng.random()
        if kind < 0.25:
            specs.append(TensorSpec(f"v{t}", int(rng.integers(0, 3000)), 1, 1))
        elif kind < 0.45:
            rows, cols = int(rng.integers(1, 300)), int(rng.integers(1, 200))
            gran = [1, 4, rows][int(rng.integers(0, 3))]
            specs.append(TensorSpec(f"m{t}", rows, cols, gran))
        else:
            qb = BLOCKS[int(rng.integers(0, len(BLOCKS)))]
            rows = int(rng.integers(0, 3 * qb[0] + 40))
            cols = int(rng.integers(1, 3 * qb[1] + 20))
            quant = "e4m3" if rng.random() < 0.5 else "int8"
            specs.append(TensorSpec(f"q{t}", rows, cols, qb[0], qblock=qb, quant=quant))
    m = int(rng.integers(1, 10))
    units = [int(u) for u in rng.integers(1, 5, m)] if rng.random() < 0.3 else None
    align = 16 if rng.random() < 0.7 else 1
    return specs, m, units, align


@pytest.mark.parametrize("seed", range(N_GROUPS))
def test_random_group_all_operators(dbuf_lib, oracle_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    specs, m, units, align = random_group(rng)
    gdt = torch.bfloat16 if rng.random() < 0.3 else torch.float32
    gen = torch.Generator().manual_seed(seed)
    params = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    full_group_parity(oracle_lib, specs, m, units, align,
                      param_fn=lambda t: params[t],
                      grad_fn=lambda t, step: (torch.randn(specs[t].rows, specs[t].cols,
                                                           generator=gen) * 1e-3).to(gdt),
                      grad_dtype=gdt, scale=1.0 / max(m, 1), accum_steps=2)


@pytest.mark.parametrize("seed", range(N_ADAMW8))
def test_random_group_adamw8(dbuf_lib, oracle_lib, seed):
    rng = np.random.default_rng(2000 + seed)
    specs, m, units, align = random_group(rng)
    c = Case(oracle_lib, specs, m, units=units, align=align, seed=seed,
             shift=1 if rng.random() < 0.2 else 0)
    c.step(1, clip=True)
    c.step(2)


# larger groups: many tensors (several quantiser and 8-bit AdamW launches),
# tiles enough for the persistent kernels' cut grids and several rounds
BIG_BLOCKS = [(128, 128), (64, 128), (32, 32), (1, 128), (128, 96), (64, 256), (256, 64)]
N_LARGE = int(os.environ.get("DBUF_LARGE_RANDOM", "0")) or 2


def large_random_group(rng):
    specs = []
    for t in range(int(rng.integers(20, 70))):
        kind = rng.random()
        if kind < 0.15:
            specs.append(TensorSpec(f"v{t}", int(rng.integers(1, 20000)), 1, 1))
        elif kind < 0.3:
            rows, cols = int(rng.integers(1, 1500)), 4 * int(rng.integers(1, 400))
            specs.append(TensorSpec(f"m{t}", rows, cols, [1, 8, rows][int(rng.integers(0, 3))]))
        else:
            qb = BIG_BLOCKS[int(rng.integers(0, len(BIG_BLOCKS)))]
            rows = int(rng.integers(1, 12)) * qb[0] + int(rng.integers(0, 3)) * 7
            cols = int(rng.integers(1, 10)) * qb[1] + int(rng.integers(0, 2)) * 20
            quant = "e4m3" if rng.random() < 0.5 else "int8"
            specs.append(TensorSpec(f"q{t}", rows, cols, qb[0], qblock=qb, quant=quant))
    m = int(rng.integers(2, 17))
    units = [int(u) for u in rng.integers(1, 4, m)] if rng.random() < 0.3 else None
    return specs, m, units, 16


@pytest.mark.parametrize("seed", range(N_LARGE))
def test_large_random_group_all_operators_and_adamw8(dbuf_lib, oracle_lib, seed):
    """Groups of 20-70 tensors up to a few million elements each: every step
    operator on whole buffers (fp32 or bf16 gradients), then two 8-bit AdamW
    steps (now and then on unaligned buffers), against the oracle."""
    rng = np.random.default_rng(4000 + seed)
    specs, m, units, align = large_random_group(rng)
    gdt = torch.bfloat16 if rng.random() < 0.3 else torch.float32
    shift = 1 if rng.random() < 0.2 else 0  # 8-bit AdamW on unaligned buffers
    gen = torch.Generator().manual_seed(4000 + seed)
    params = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    full_group_parity(oracle_lib, specs, m, units, align,
                      param_fn=lambda t: params[t],
                      grad_fn=lambda t, step: (torch.randn(specs[t].rows, specs[t].cols,
                                                           generator=gen) * 1e-3).to(gdt),
                      grad_dtype=gdt, scale=1.0 / m, accum_steps=1)
    c = Case(oracle_lib, specs, m, units=units, align=align, seed=seed, shift=shift)
    c.step(1, clip=True)
    c.step(2)
