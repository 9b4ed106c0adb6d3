"""dbuf_norm_nonfinite_noalloc: the norm / non-finite check for callers that
cannot allocate device memory (a host program whose framework already holds the
device memory in its own pool, or an out-of-memory recovery path that still has
to look for inf/NaN gradients).  It uses the library's static scratch instead of
a caller workspace.  Checked through the C ABI against the workspace entry point
on consecutive calls; this file is collected last so that a failing run that
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _outs(n):
    return (torch.empty(max(n, 1), dtype=torch.float32, device=DEV),
            torch.empty(1, dtype=torch.float32, device=DEV),
            torch.empty(1, dtype=torch.int32, device=DEV))


def _noalloc(d, db, buf, out):
    dt = d.DBUF_F32 if buf.dtype == torch.float32 else d.DBUF_BF16
    d.dbuf_norm_nonfinite_noalloc(db.handle, buf.data_ptr(), dt, out[0].data_ptr(),
                                  out[1].data_ptr(), out[2].data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out[0][:db.n].cpu().numpy().astype(np.float64), float(out[1].item()), int(out[2].item())


def _with_workspace(db, buf):
    norms, total, flag = db.norm_nonfinite(buf)
    torch.cuda.synchronize()
    return norms.cpu().numpy().astype(np.float64), float(total.item()), int(flag.item())


def _close(a, b, rel=1e-5):
    na, ta, fa = a
    nb, tb, fb = b
    assert fa == fb
    if fa == 0:
        assert np.all(np.abs(na - nb) <= rel * np.abs(nb))
        assert abs(ta - tb) <= rel * abs(tb)


def test_noalloc_norm_matches_workspace_entry_point(dbuf_lib):
    from fsdp_infra_gb300 import DBuffer
    from workloads import workload, grad_values
    d = dbuf_lib
    w = workload("llama_layer")
    specs = w.groups[0].tensors
    db = DBuffer(specs, w.m, None, w.align).upload()
    assert d.dbuf_workspace_bytes(db.handle, d.DBUF_OP_NORM_NONFINITE) <= d.DBUF_NOALLOC_SCRATCH_BYTES
    buf = torch.zeros(db.total, dtype=torch.float32, device=DEV)
    out = _outs(db.n)
    # consecutive calls on different data: the second must not see the first's scratch
    for call, seed in enumerate([3, 4]):
        for t, s in enumerate(specs):
            buf[db.offsets[t]:db.offsets[t] + s.numel].copy_(
                grad_values(w, 0, t, seed=seed, device=DEV).reshape(-1))
        got = _noalloc(d, db, buf, out)
        want = _with_workspace(db, buf)
        assert got[2] == 0
        _close(got, want)
    # a non-finite value raises the flag, and clearing it lowers the flag again
    o = db.offsets[2] + 12345
    buf[o] = float("inf")
    assert _noalloc(d, db, buf, out)[2] == 1 == _with_workspace(db, buf)[2]
    buf[o] = 0.0
    _close(_noalloc(d, db, buf, out), _with_workspace(db, buf))
    # a bf16 buffer
    b16 = buf.to(torch.bfloat16)
    _close(_noalloc(d, db, b16, out), _with_workspace(db, b16))
    db.close()


def test_noalloc_norm_rejects_plans_beyond_its_scratch(dbuf_lib):
    """A plan whose norm needs more scratch than the static array is refused
    before anything runs."""
    from fsdp_infra_gb300 import DBuffer
    d = dbuf_lib
    db = DBuffer([(1 << 31, 1, 1)], 1).upload()
    assert d.dbuf_workspace_bytes(db.handle, d.DBUF_OP_NORM_NONFINITE) > d.DBUF_NOALLOC_SCRATCH_BYTES
    small = torch.zeros(16, dtype=torch.float32, device=DEV)
    out = _outs(1)
    with pytest.raises(d.DbufError) as e:
        d.dbuf_norm_nonfinite_noalloc(db.handle, small.data_ptr(), d.DBUF_F32, out[0].data_ptr(),
                                      out[1].data_ptr(), out[2].data_ptr(), 0)
    assert e.value.code == d.DBUF_ERANGE
    db.close()
