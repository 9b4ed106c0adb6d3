"""One plan shared by host threads, each on its own stream.

The boundary promises that a plan is immutable after upload and may be
shared across host threads.  Four Python threads (the library's calls release
the interpreter lock) each take their own CUDA stream, buffers and norm
workspace on the same DBuffer objects and run the step's operators and the
8-bit AdamW step three times; every thread's results must equal, bit for bit,
the same sequence run alone on one stream.
"""
import threading

import numpy as np
import pytest
import torch

from workloads.configs import TensorSpec

from gpu_helpers import assert_bits_equal, f32

pytestmark = pytest.mark.gpu

DEV = "cuda"
THREADS, ROUNDS = 4, 3

SPECS = [
    TensorSpec("wqkv", 512, 384, 128, qblock=(128, 128), quant="e4m3"),
    TensorSpec("norm", 384, 1, 0, kind="norm"),
    TensorSpec("w_row", 96, 640, 1, qblock=(1, 128), quant="int8"),
    TensorSpec("bias", 200, 1, 1),
    TensorSpec("wo", 384, 384, 128, qblock=(128, 128), quant="e4m3"),
]
SPECS8 = [
    TensorSpec("a", 320, 256, 32, qblock=(32, 32), quant="int8"),
    TensorSpec("v", 96, 1, 1),
    TensorSpec("b", 160, 384, 32, qblock=(32, 32), quant="int8"),
]


def _inputs(seed):
    g = torch.Generator().manual_seed(seed)
    params = [torch.randn(s.rows, s.cols, generator=g) * 0.02 for s in SPECS]
    grads = [torch.randn(s.numel, generator=g) * 1e-3 for s in SPECS]
    p8 = [torch.randn(s.numel, generator=g) * 0.02 for s in SPECS8]
    g8 = [torch.randn(s.numel, generator=g) * 1e-3 for s in SPECS8]
    return params, grads, p8, g8


def _run(db, db8, inputs, stream):
    """The operator sequence on `stream`; returns host copies of every output."""
    params, grads, p8, g8 = inputs
    with torch.cuda.stream(stream):
        src = [p.to(DEV, non_blocking=False) for p in params]
        buf16 = torch.zeros(db.total, dtype=torch.bfloat16, device=DEV)
        dst = [torch.empty(s.rows, s.cols, dtype=torch.bfloat16, device=DEV) for s in SPECS]
        grad = torch.zeros(db.total, dtype=torch.float32, device=DEV)
        acc = torch.zeros(db.total, dtype=torch.float32, device=DEV)
        ws = db.new_workspace()
        P = torch.zeros(db8.total, dtype=torch.float32, device=DEV)
        G = torch.zeros(db8.total, dtype=torch.float32, device=DEV)
        for t, s in enumerate(SPECS8):
            P[db8.offsets[t]:db8.offsets[t] + s.numel].copy_(p8[t])
            G[db8.offsets[t]:db8.offsets[t] + s.numel].copy_(g8[t])
        st8 = db8.new_adamw8_state()
        out8 = db8.norm_nonfinite(G, stream=stream, workspace=db8.new_workspace())
        for r in range(ROUNDS):
            for t, s in enumerate(SPECS):
                grad[db.offsets[t]:db.offsets[t] + s.numel].copy_(grads[t] * (r + 1))
            db.pack_cast(src, buf16, stream=stream)
            db.unpack(buf16, dst, stream=stream)
            db.scale_accum_zero(grad, acc, 0.25, stream=stream)
            norms, total, flag = db.norm_nonfinite(acc, stream=stream, workspace=ws)
            codes, scales = db.block_quant(acc, stream=stream)
            db8.adamw8_step(P, G, st8, step=r + 1, lr=1e-3, betas=(0.9, 0.95), eps=1e-8,
                            weight_decay=0.1, max_norm=0.5, total_norm=out8[1],
                            nonfinite=out8[2], stream=stream)
        stream.synchronize()
        return {"buf16": buf16.view(torch.int16).cpu().numpy(),
                "dst": [d.view(torch.int16).cpu().numpy() for d in dst],
                "acc": f32(acc), "grad": f32(grad), "norms": f32(norms), "total": f32(total),
                "flag": int(flag.item()), "codes": codes.cpu().numpy(), "scales": f32(scales),
                "P": f32(P), "mc": st8["m_codes"].cpu().numpy(), "vc": st8["v_codes"].cpu().numpy(),
                "ms": f32(st8["m_scales"]), "vs": f32(st8["v_scales"]), "m32": f32(st8["m32"]),
                "v32": f32(st8["v32"])}


def _same(a, b, what):
    for k in a:
        if isinstance(a[k], list):
            for i, (x, y) in enumerate(zip(a[k], b[k])):
                assert np.array_equal(x, y), f"{what}: {k}[{i}] differs"
        elif isinstance(a[k], np.ndarray) and a[k].dtype == np.float32:
            assert_bits_equal(a[k], b[k], f"{what}: {k}")
        else:
            assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), f"{what}: {k} differs"


def test_one_plan_shared_by_threads_on_their_own_streams(dbuf_lib):
    from fsdp_infra_gb300 import DBuffer
    db = DBuffer(SPECS, 4).upload()
    db8 = DBuffer(SPECS8, 4).upload()
    inputs = [_inputs(100 + i) for i in range(THREADS)]
    want = [_run(db, db8, inputs[i], torch.cuda.Stream()) for i in range(THREADS)]
    got = [None] * THREADS
    errors = []

    def work(i):
        try:
            got[i] = _run(db, db8, inputs[i], torch.cuda.Stream())
        except Exception as e:  # reported on the main thread
            errors.append((i, e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(THREADS):
        _same(want[i], got[i], f"thread {i}")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0 and dbuf.dbuf_device_status(db8.handle) == 0
