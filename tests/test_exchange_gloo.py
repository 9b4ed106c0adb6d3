"""The exchange around the group operators (fsdp_infra_gb300.exchange) on two
gloo ranks on the CPU, with the oracle as each rank's compute.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer and
Figure 7 (AllGather of parameters and ReduceScatter of gradients in place on the
flat buffer, one slice per rank); "PyTorch FSDP: Experiences on Scaling Fully
Sharded Data Parallel", FlatParameter (equal shard sizes).

Each rank runs ShardedStep (the product's exchange) with shims whose operators
are the oracle's, applied to the full plan and to the rank's slice.  The slice
geometry in the shims is computed here from the oracle's layout (a tensor's
piece in slice k is its range intersected with [B_k, B_{k+1})).  The result of
both ranks is compared with one oracle run over the whole buffer: the summed
gradients of both ranks accumulated with scale 1/2, the norms of the whole
accumulator, its block quantisation, and the parameters' copy-in and copy-out.
With two ranks the gradient sum has one rounding in either order, so the
accumulator, codes, scales and compute tensors must agree bit for bit; the norms
within 1e-5 (partial sums are added in another order).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _specs():
    from workloads.configs import TensorSpec
    return [TensorSpec("wq", 96, 64, 32, (32, 32), "e4m3"),
            TensorSpec("norm", 64, 1, 1),
            TensorSpec("w1", 64, 160, 32, (32, 32), "e4m3"),
            TensorSpec("bias", 37, 1, 1),
            TensorSpec("rows", 48, 32, 1, (1, 16), "int8"),
            TensorSpec("whole", 7, 9, 0),
            TensorSpec("empty", 0, 4, 1)]


M, ALIGN = 2, 16


def _host(t: torch.Tensor) -> np.ndarray:
    """A numpy view sharing the tensor's memory, in the oracle's representation."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class OracleFull:
    """The full plan's operators as the oracle computes them."""

    def __init__(self, oracle, specs, op):
        self.o, self.specs, self.op = oracle, specs, op
        self.m = len(op.bounds) - 1
        self.shard_bounds = [int(b) for b in op.bounds]
        self.S, self.total = op.S, op.total

    def pack_cast(self, srcs, buf):
        self.o.pack(self.op, [s.reshape(-1).numpy() for s in srcs], _host(buf))

    def unpack(self, buf, dsts):
        self.o.unpack(self.op, _host(buf), [_host(d).reshape(-1) for d in dsts])


class OracleSlice:
    """Slice k's operators: the oracle applied to the pieces inside the slice."""

    def __init__(self, oracle, specs, op, k):
        from workloads.configs import TensorSpec
        self.o = oracle
        B0, B1 = int(op.bounds[k]), int(op.bounds[k + 1])
        self.total = self.S = B1 - B0
        self.src, offs, num, self.pspecs = [], [], [], []
        for t, s in enumerate(specs):
            l = int(op.offsets[t])
            lo, hi = max(l, B0), min(l + s.numel, B1)
            n = max(0, hi - lo)
            self.src.append(lo - l if n else 0)
            offs.append(lo - B0 if n else 0)
            num.append(n)
            rows = n // s.cols if s.quant else n
            self.pspecs.append(TensorSpec(s.name, rows, s.cols if s.quant else 1, 0, s.qblock,
                                          s.quant))
        self.plan = oracle.Plan(self.S, np.array(offs, np.int64), np.array([0, self.S], np.int64),
                                np.array(num, np.int64))
        self.n_scales = oracle.scale_offsets(self.pspecs)[1]

    def pack_cast(self, srcs, buf):
        pieces = [s.reshape(-1).numpy()[a:a + n] for s, a, n in zip(srcs, self.src,
                                                                      self.plan.numel)]
        self.o.pack(self.plan, pieces, _host(buf))

    def scale_accum_zero(self, grad, acc, scale):
        self.o.scale_accum_zero(self.plan, _host(grad), _host(acc), scale)

    def norm_sumsq(self, acc):
        norms, _, flag = self.o.norm_nonfinite(self.plan, _host(acc))
        return (torch.from_numpy(np.asarray(norms, np.float64) ** 2),
                torch.tensor([flag], dtype=torch.int32))

    def norm_finish(self, sumsq):
        s = sumsq.numpy()
        return (torch.from_numpy(np.sqrt(s).astype(np.float32)),
                torch.tensor([np.sqrt(np.sum(s))], dtype=torch.float32))

    def block_quant(self, acc, codes=None, scales=None):
        c = np.zeros(self.total, np.uint8)
        sc = self.o.block_quant(self.plan, self.pspecs, _host(acc), c)
        return torch.from_numpy(c), torch.from_numpy(sc)


def _inputs(specs, rank, inf=False):
    gen = torch.Generator().manual_seed(5)
    master = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
    gen = torch.Generator().manual_seed(100 + rank)
    grads = [torch.randn(s.rows, s.cols, generator=gen) * 1e-3 for s in specs]
    if inf and rank == 1:
        grads[2][5, 7] = float("inf")
    gen = torch.Generator().manual_seed(77)
    acc0 = torch.randn(M * 100000, generator=gen) * 1e-3   # cut to the buffer size below
    return master, grads, acc0


def _worker(rank, world, port, q, inf):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path[:0] = [ROOT, HERE]
    import torch.distributed as dist
    import oracle
    from fsdp_infra_gb300.exchange import ShardedStep
    dist.init_process_group("gloo", rank=rank, world_size=world)
    specs = _specs()
    op = oracle.plan_specs(specs, M, None, ALIGN)
    full, local = OracleFull(oracle, specs, op), OracleSlice(oracle, specs, op, rank)
    step = ShardedStep(full, local, rank, world)
    master, grads, acc0 = _inputs(specs, rank, inf)
    S = op.S
    grad_full = torch.zeros(op.total, dtype=torch.float32)
    grad_local = torch.zeros(S, dtype=torch.float32)
    acc_local = acc0[rank * S:(rank + 1) * S].clone()
    norms, total, flag, codes, scales = step.reduce_gradients(grads, grad_full, grad_local,
                                                              acc_local, 1.0 / world)
    buf_local = torch.zeros(S, dtype=torch.bfloat16)
    buf_full = torch.zeros(op.total, dtype=torch.bfloat16)
    compute = [torch.zeros(s.rows, s.cols, dtype=torch.bfloat16) for s in specs]
    step.gather_parameters(master, buf_local, buf_full, compute)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, acc_local.numpy().copy(), grad_local.numpy().copy(), norms.numpy().copy(),
           float(total[0]), int(flag[0]), None if codes is None else codes.numpy().copy(),
           None if scales is None else scales.numpy().copy(),
           [_host(c).reshape(-1).copy() for c in compute]))


def _run(inf):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, M, port, q, inf)) for r in range(M)]
    for p in procs:
        p.start()
    out = []
    import queue
    import time
    deadline = time.time() + 300
    while len(out) < M:
        try:
            out.append(q.get(timeout=1))
        except queue.Empty:
            assert all(p.exitcode in (None, 0) for p in procs), [p.exitcode for p in procs]
            assert time.time() < deadline, "ranks did not finish"
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return sorted(out, key=lambda x: x[0])


def _reference(oracle_lib, inf):
    specs = _specs()
    op = oracle_lib.plan_specs(specs, M, None, ALIGN)
    total = op.total
    summed = np.zeros(total, np.float32)
    for r in range(M):
        master, grads, acc0 = _inputs(specs, r, inf)
        g = np.zeros(total, np.float32)
        oracle_lib.pack(op, [x.reshape(-1).numpy() for x in grads], g)
        summed = summed + g
    acc = acc0[:total].numpy().copy()
    oracle_lib.scale_accum_zero(op, summed, acc, 1.0 / M)
    norms, tot, flag = oracle_lib.norm_nonfinite(op, acc)
    codes = np.zeros(total, np.uint8)
    scales = oracle_lib.block_quant(op, specs, acc, codes)
    b16 = np.zeros(total, np.uint16)
    oracle_lib.pack(op, [x.reshape(-1).numpy() for x in master], b16)
    comp = [np.zeros(s.numel, np.uint16) for s in specs]
    oracle_lib.unpack(op, b16, comp)
    return op, acc, summed, norms, tot, flag, codes, scales, comp


def test_exchange_on_two_gloo_ranks_equals_one_buffer(oracle_lib):
    op, acc, summed, norms, tot, flag, codes, scales, comp = _reference(oracle_lib, False)
    assert flag == 0
    n_seen = 0
    for rank, acc_l, grad_l, norms_l, tot_l, flag_l, codes_l, scales_l, comp_l in _run(False):
        B0, B1 = int(op.bounds[rank]), int(op.bounds[rank + 1])
        assert np.array_equal(acc_l.view(np.uint32), acc[B0:B1].view(np.uint32))
        assert np.array_equal(grad_l.view(np.uint32), summed[B0:B1].view(np.uint32))
        assert flag_l == 0
        assert np.all(np.abs(norms_l - norms) <= 1e-5 * norms)
        assert abs(tot_l - tot) <= 1e-5 * tot
        assert codes_l is not None
        assert np.array_equal(codes_l, codes[B0:B1])
        assert np.array_equal(scales_l.view(np.uint32),
                              scales[n_seen:n_seen + scales_l.size].view(np.uint32))
        n_seen += scales_l.size
        for c, w in zip(comp_l, comp):
            assert np.array_equal(c, w)
    assert n_seen == scales.size


def test_exchange_flags_an_inf_on_one_rank_everywhere(oracle_lib):
    out = _run(True)
    assert [x[5] for x in out] == [1, 1]
