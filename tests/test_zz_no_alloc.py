"""dbuf_norm_nonfinite_noalloc: the norm / non-finite check for callers that
cannot allocate device memory (a host program whose framework already holds the
device memory in its own pool, or an out-of-memory recovery path that still has
to look for inf/NaN gradients).  It uses the library's static scratch array
instead of a caller workspace, and runs the same kernel, so its results must
equal those of dbuf_norm_nonfinite bit for bit; both are also checked against
the oracle (1e-5 relative).

Calls alternate between two plans of different sizes (the Llama layer, 7
tensors, and a 41-tensor ragged group with empty tensors and uneven shards), two
calls in a row on each, so a call that found the previous plan's completion
counters or partial sums in the array would show up.  This file is collected
last so that a failing run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import random

import numpy as np
import pytest
import torch

from gpu_helpers import assert_norms_close, host_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _outs(n):
    return (torch.empty(max(n, 1), dtype=torch.float32, device=DEV),
            torch.empty(1, dtype=torch.float32, device=DEV),
            torch.empty(1, dtype=torch.int32, device=DEV))


def _noalloc(d, db, buf, out):
    dt = d.DBUF_F32 if buf.dtype == torch.float32 else d.DBUF_BF16
    out[0].fill_(-1.0)
    out[1].fill_(-1.0)
    out[2].fill_(-1)
    d.dbuf_norm_nonfinite_noalloc(db.handle, buf.data_ptr(), dt, out[0].data_ptr(),
                                  out[1].data_ptr(), out[2].data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return (out[0][:db.n].cpu().numpy().copy(), out[1].cpu().numpy().copy(),
            int(out[2].item()))


def _with_workspace(db, buf):
    norms, total, flag = db.norm_nonfinite(buf)
    torch.cuda.synchronize()
    return norms.cpu().numpy().copy(), total.cpu().numpy().copy(), int(flag.item())


def _bitwise(got, want):
    assert got[2] == want[2]
    assert np.array_equal(got[0].view(np.uint32), want[0].view(np.uint32))
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def _against_oracle(oracle_lib, case, buf, got):
    wn, wt, wf = oracle_lib.norm_nonfinite(case["op"], host_bits(buf))
    assert got[2] == wf
    if wf == 0:
        assert_norms_close(got[0], float(got[1][0]), wn, wt, what="noalloc norms")


def _ragged_specs():
    from workloads.configs import TensorSpec
    rng = random.Random(5)
    specs = []
    for i in range(41):
        if i % 4 == 1:
            specs.append(TensorSpec(f"empty{i}", 0, rng.randint(1, 64), 1))
        elif i % 4 == 2:
            specs.append(TensorSpec(f"vec{i}", rng.randint(1, 5000), 1, 1))
        else:
            r, c = rng.randint(1, 300), rng.choice([16, 48, 100, 256])
            specs.append(TensorSpec(f"mat{i}", r, c, rng.choice([0, 1, 4])))
    return specs


def _cases(oracle_lib):
    from fsdp_infra_gb300 import DBuffer
    from workloads import workload
    w = workload("llama_layer")
    ragged = _ragged_specs()
    units = [1, 3, 2, 1, 2]
    return [
        {"name": "llama_layer", "specs": w.groups[0].tensors,
         "db": DBuffer(w.groups[0].tensors, w.m, None, w.align).upload(),
         "op": oracle_lib.plan_specs(w.groups[0].tensors, w.m, None, w.align)},
        {"name": "ragged", "specs": ragged, "db": DBuffer(ragged, 5, units, 16).upload(),
         "op": oracle_lib.plan_specs(ragged, 5, units, 16)},
    ]


def _fill(case, seed, dtype=torch.float32):
    db = case["db"]
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    for t, s in enumerate(case["specs"]):
        if s.numel:
            o = db.offsets[t]
            buf[o:o + s.numel].normal_(0.0, 1e-3, generator=gen)
    return buf.to(dtype)


def test_noalloc_norm_equals_workspace_entry_point(dbuf_lib, oracle_lib):
    d = dbuf_lib
    cases = _cases(oracle_lib)
    for c in cases:
        assert c["db"].offsets == [int(x) for x in c["op"].offsets]
        assert (d.dbuf_workspace_bytes(c["db"].handle, d.DBUF_OP_NORM_NONFINITE)
                <= d.DBUF_NOALLOC_SCRATCH_BYTES)
    seed = 100
    # two calls in a row on each plan, alternating plans: A A B B A A B B
    for rnd in range(2):
        for c in cases:
            out = _outs(c["db"].n)
            for _ in range(2):
                seed += 1
                buf = _fill(c, seed)
                got = _noalloc(d, c["db"], buf, out)
                assert got[2] == 0
                _bitwise(got, _with_workspace(c["db"], buf))
                _against_oracle(oracle_lib, c, buf, got)
    # a non-finite value raises the flag on one plan; the next call on the
    # other plan, and the same plan cleared again, come back clean
    a, b = cases
    buf = _fill(a, 7)
    buf[a["db"].offsets[2] + 12345] = float("inf")
    out_a, out_b = _outs(a["db"].n), _outs(b["db"].n)
    got = _noalloc(d, a["db"], buf, out_a)
    assert got[2] == 1
    _bitwise(got, _with_workspace(a["db"], buf))
    bbuf = _fill(b, 8)
    got = _noalloc(d, b["db"], bbuf, out_b)
    assert got[2] == 0
    _bitwise(got, _with_workspace(b["db"], bbuf))
    buf[a["db"].offsets[2] + 12345] = 0.0
    got = _noalloc(d, a["db"], buf, out_a)
    _bitwise(got, _with_workspace(a["db"], buf))
    _against_oracle(oracle_lib, a, buf, got)
    # bf16 buffers
    for c in cases:
        b16 = _fill(c, 9, torch.bfloat16)
        got = _noalloc(d, c["db"], b16, _outs(c["db"].n))
        _bitwise(got, _with_workspace(c["db"], b16))
        _against_oracle(oracle_lib, c, b16, got)
    # empty tensors report a zero norm
    for t, s in enumerate(b["specs"]):
        if s.numel == 0:
            assert got[0][t] == 0.0
    for c in cases:
        c["db"].close()


def test_noalloc_norm_rejects_plans_beyond_its_scratch(dbuf_lib):
    """A plan whose norm needs more scratch than the static array is refused
    before anything runs."""
    from fsdp_infra_gb300 import DBuffer
    d = dbuf_lib
    db = DBuffer([(1, 1, 1)] * 8200, 1).upload()  # 128 bytes of counters per tensor
    assert d.dbuf_workspace_bytes(db.handle, d.DBUF_OP_NORM_NONFINITE) > d.DBUF_NOALLOC_SCRATCH_BYTES
    small = torch.zeros(16, dtype=torch.float32, device=DEV)
    out = _outs(1)
    with pytest.raises(d.DbufError) as e:
        d.dbuf_norm_nonfinite_noalloc(db.handle, small.data_ptr(), d.DBUF_F32, out[0].data_ptr(),
                                      out[1].data_ptr(), out[2].data_ptr(), 0)
    assert e.value.code == d.DBUF_ERANGE
    db.close()
