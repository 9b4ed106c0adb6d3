"""The bounded device-side waits end in an error status, not a hang: a CTA
that waits on an mbarrier phase nothing completes gives up after its limit and
records DBUF_ETIMEOUT in the plan's status word; the host reads it back (and
clears it), and the context keeps working."""
import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_runs_out_reports_timeout(dbuf_lib, oracle_lib):
    from fsdp_infra_gb300 import DBuffer
    d = dbuf_lib
    specs = [TensorSpec("a", 64, 64, 32, (32, 32), "int8"), TensorSpec("v", 40, 1, 1)]
    db = DBuffer(specs, 2, None, 16).upload()
    assert d.dbuf_device_status(db.handle) == 0
    for tries in (1, 1000):
        d.dbuf_selftest_wait_timeout(db.handle, tries)
        assert d.dbuf_device_status(db.handle) == d.DBUF_ETIMEOUT
        assert d.dbuf_device_status(db.handle) == 0          # reading clears it
    for bad in (0, (1 << 22) + 1):
        with pytest.raises(d.DbufError) as e:
            d.dbuf_selftest_wait_timeout(db.handle, bad)
        assert e.value.code == d.DBUF_EINVAL
    # the context is intact: an operator still runs and matches the oracle
    op = oracle_lib.plan_specs(specs, 2, None, 16)
    gen = torch.Generator().manual_seed(3)
    host = (torch.randn(db.total, generator=gen) * 0.1).to(torch.float32)
    codes, scales = db.block_quant(host.to(DEV))
    want_c = np.zeros(db.total, np.uint8)
    want_s = oracle_lib.block_quant(op, specs, host.numpy().copy(), want_c)
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    rng = [(int(o), s.numel) for o, s in zip(op.offsets, specs) if s.quant]
    for o, n in rng:
        assert np.array_equal(codes.cpu().numpy()[o:o + n], want_c[o:o + n])
    assert d.dbuf_device_status(db.handle) == 0
    db.close()
