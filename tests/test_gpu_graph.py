"""The step's operators captured once in a CUDA graph and replayed, as the
benchmark times them, against the oracle on every replay.

Inside a graph the kernels run as programmatic dependents of one another, the
norm's workspace and completion counters are reused from one replay to the
next, and the user tensors are the same allocations every time with new values
copied in between replays.  Each replay must still give the oracle's results:
pack (fp32 -> bf16), unpack (bf16 -> bf16), scale/accumulate/zero (the
accumulator carried across replays), norms and flag, block codes and scales, and
a fused AdamW step on the accumulated gradients.  A replay with an inf in one
tensor raises the flag, and the next clean replay clears it.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_norms_close, bf16_bits, f32, host_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _ragged_quant_specs():
    """Tensors for the three quantisers: tiles the tensor maps fetch (128x128 and
    2x100 blocks), row blocks (1x128), and tiles they cannot (4x35: rows of 35
    elements), between vectors and unquantised matrices."""
    from workloads.configs import TensorSpec
    return [TensorSpec("a", 256, 384, 128, qblock=(128, 128), quant="e4m3"),
            TensorSpec("v", 1000, 1, 1),
            TensorSpec("b", 200, 136, 8, qblock=(1, 128), quant="int8"),
            TensorSpec("c", 130, 100, 2, qblock=(2, 100), quant="e4m3"),
            TensorSpec("d", 60, 70, 4, qblock=(4, 35), quant="int8"),  # the register-tile kernel
            TensorSpec("w", 77, 64, 1)]


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_step_replayed_from_a_cuda_graph_matches_the_oracle(dbuf_lib, oracle_lib, case):
    from fsdp_infra_gb300 import DBuffer
    from workloads import workload
    if case == "tiny":
        w = workload("tiny")
        specs, m, units, align, scale = w.groups[0].tensors, w.m, None, w.align, w.scale
    else:
        specs, m, units, align, scale = _ragged_quant_specs(), 3, [2, 1, 3], 16, 1.0 / 3
    n = len(specs)
    op = oracle_lib.plan_specs(specs, m, units, align)
    db = DBuffer(specs, m, units, align).upload()
    assert db.offsets == [int(x) for x in op.offsets]
    total = db.total

    # static buffers: the graph reads and writes these same allocations every replay
    params = [torch.zeros(s.rows, s.cols, dtype=torch.float32, device=DEV) for s in specs]
    compute = [torch.zeros(s.rows, s.cols, dtype=torch.bfloat16, device=DEV) for s in specs]
    buf16 = torch.zeros(total, dtype=torch.bfloat16, device=DEV)
    grad = torch.zeros(total, dtype=torch.float32, device=DEV)
    acc = torch.zeros(total, dtype=torch.float32, device=DEV)
    codes = torch.full((total,), 0x5A, dtype=torch.uint8, device=DEV)
    scales = torch.zeros(max(db.n_scales, 1), dtype=torch.float32, device=DEV)
    outs = (torch.zeros(max(n, 1), dtype=torch.float32, device=DEV),
            torch.zeros(1, dtype=torch.float32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))
    p32 = torch.zeros(total, dtype=torch.float32, device=DEV)
    m32 = torch.zeros(total, dtype=torch.float32, device=DEV)
    v32 = torch.zeros(total, dtype=torch.float32, device=DEV)
    hp = dict(step=3, lr=1e-3, betas=(0.9, 0.95), weight_decay=0.1, max_norm=1.0, eps=1e-8)

    def step():
        db.pack_cast(params, buf16)
        db.unpack(buf16, compute)
        db.scale_accum_zero(grad, acc, scale)
        norms, tot, flag = db.norm_nonfinite(acc, out=outs)
        db.block_quant(acc, codes=codes, scales=scales)
        db.adamw_step(p32, acc, m32, v32, total_norm=tot, nonfinite=flag, **hp)

    # one eager pass builds the pointer tables and the workspace outside the capture
    step()
    torch.cuda.synchronize()
    acc.zero_()
    codes.fill_(0x5A)
    p32.zero_()
    m32.zero_()
    v32.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    gen = torch.Generator().manual_seed(71)
    acc_h = np.zeros(total, np.float32)
    want_codes = np.full(total, 0x5A, np.uint8)
    p_h = (torch.randn(total, generator=gen) * 0.02).numpy().astype(np.float32)
    m_h = np.zeros(total, np.float32)
    v_h = np.zeros(total, np.float32)
    p32.copy_(torch.from_numpy(p_h))
    for r in range(4):
        pv = [torch.randn(s.rows, s.cols, generator=gen) * 0.02 for s in specs]
        gh = np.zeros(total, np.float32)
        for t, s in enumerate(specs):
            o = db.offsets[t]
            gh[o:o + s.numel] = (torch.randn(s.numel, generator=gen) * 1e-3).numpy()
        inf_at = None
        if r == 2:  # a non-finite gradient: the flag, then a clean replay clears it
            inf_at = db.offsets[n - 1] + 5
            gh[inf_at] = np.inf
        for t in range(n):
            params[t].copy_(pv[t])
        grad.copy_(torch.from_numpy(gh))
        graph.replay()
        torch.cuda.synchronize()

        want16 = np.zeros(total, np.uint16)
        oracle_lib.pack(op, [f32(x) for x in pv], want16)
        got16 = bf16_bits(buf16)
        for t, s in enumerate(specs):
            o = db.offsets[t]
            assert_bits_equal(got16[o:o + s.numel], want16[o:o + s.numel], f"pack, replay {r}")
            assert_bits_equal(bf16_bits(compute[t]).reshape(-1), want16[o:o + s.numel],
                              f"unpack, replay {r}")
        oracle_lib.scale_accum_zero(op, gh, acc_h, scale)
        assert_bits_equal(host_bits(grad), gh, f"gradient zeroed, replay {r}")
        assert_bits_equal(f32(acc), acc_h, f"accumulator, replay {r}")
        wn, wt, wf = oracle_lib.norm_nonfinite(op, acc_h)
        assert int(outs[2].item()) == wf == (1 if inf_at is not None else 0), r
        if wf:
            # a skipped step: the moments and parameters keep their values; the
            # accumulator is reset for the next replays, as a scaler would
            assert np.array_equal(f32(p32).view(np.uint32), p_h.view(np.uint32))
            assert np.array_equal(f32(m32).view(np.uint32), m_h.view(np.uint32))
            assert np.array_equal(f32(v32).view(np.uint32), v_h.view(np.uint32))
            acc.zero_()
            acc_h[:] = 0.0
            continue
        assert_norms_close(f32(outs[0])[:n], float(outs[1].item()), wn, wt,
                           what=f"norms, replay {r}")
        ws = oracle_lib.block_quant(op, specs, acc_h, want_codes)
        assert_bits_equal(f32(scales)[:db.n_scales], ws, f"scales, replay {r}")
        assert_bits_equal(codes.cpu().numpy(), want_codes, f"codes, replay {r}")
        # the AdamW step clips with the device norm it was given
        oracle_lib.adamw(op, p_h, acc_h, m_h, v_h, lr=hp["lr"], beta1=hp["betas"][0],
                         beta2=hp["betas"][1], eps=hp["eps"], weight_decay=hp["weight_decay"],
                         step=hp["step"], max_norm=hp["max_norm"],
                         total_norm=float(outs[1].item()), nonfinite=0)
        assert_bits_equal(f32(p32), p_h, f"AdamW parameters, replay {r}")
        assert_bits_equal(f32(m32), m_h, f"AdamW first moment, replay {r}")
        assert_bits_equal(f32(v32), v_h, f"AdamW second moment, replay {r}")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0
    db.close()


def test_adamw8_and_gather_scatter_replayed_from_a_cuda_graph(dbuf_lib, oracle_lib):
    """The next rows in a graph: an 8-bit AdamW step (the stage kernel on 32x32
    blocks, the big-block kernel on 128x128, the register kernel on 128x96,
    compact fp32 moments for a vector), then the whole-matrix gather of the
    updated parameters and their scatter into a second set of shard buffers.
    Replayed three times with new gradients, clipping to a device norm that
    changes between replays; every replay bit-exact against the oracle."""
    from fsdp_infra_gb300 import DBuffer
    from workloads.configs import TensorSpec
    specs = [TensorSpec("w_sq", 96, 96, 32, qblock=(32, 32), quant="int8"),
             TensorSpec("bias", 57, 1, 1),
             TensorSpec("w_big", 256, 256, 128, qblock=(128, 128), quant="int8"),
             TensorSpec("w_reg", 128, 96, 128, qblock=(128, 96), quant="int8")]
    m, align = 4, 16
    hp = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    op = oracle_lib.plan_specs(specs, m, None, align)
    db = DBuffer(specs, m, None, align).upload()
    assert db.offsets == [int(x) for x in op.offsets]
    total, B = db.total, db.shard_bounds
    rng = np.random.default_rng(5)
    p_h = (rng.standard_normal(total) * 0.02).astype(np.float32)
    p = torch.from_numpy(p_h.copy()).to(DEV)
    g = torch.zeros(total, dtype=torch.float32, device=DEV)
    st = db.new_adamw8_state()
    ns, nst = max(db.n_scales, 1), max(db.n_state, 1)
    h = {"mc": np.zeros(total, np.uint8), "vc": np.zeros(total, np.uint8),
         "ms": np.zeros(ns, np.float32), "vs": np.zeros(ns, np.float32),
         "m32": np.zeros(nst, np.float32), "v32": np.zeros(nst, np.float32)}
    keys = {"mc": "m_codes", "vc": "v_codes", "ms": "m_scales", "vs": "v_scales",
            "m32": "m32", "v32": "v32"}
    norm = torch.zeros(1, dtype=torch.float32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    shards = [p[B[k]:B[k + 1]] for k in range(m)]
    back = torch.full((total,), -1.0, dtype=torch.float32, device=DEV)
    back_shards = [back[B[k]:B[k + 1]] for k in range(m)]
    mats = [torch.zeros(s.numel, dtype=torch.float32, device=DEV) for s in specs]

    def step():
        db.adamw8_step(p, g, st, step=4, max_norm=1e-3, total_norm=norm, nonfinite=flag, **hp)
        db.gather(shards, mats)
        db.scatter(mats, back_shards)

    # pointer tables built outside the capture; the eager pass is then undone
    saved = {k: v.clone() for k, v in st.items()}
    step()
    torch.cuda.synchronize()
    p.copy_(torch.from_numpy(p_h))
    for k, v in saved.items():
        st[k].copy_(v)
    back.fill_(-1.0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    back_h = np.full(total, -1.0, np.float32)
    for r in range(3):
        gh = (rng.standard_normal(total) * 1e-3).astype(np.float32)
        _, wt, _ = oracle_lib.norm_nonfinite(op, gh)
        tot32 = float(np.float32(wt * (0.5 + r)))  # a device norm that changes every replay
        g.copy_(torch.from_numpy(gh))
        norm.fill_(tot32)
        graph.replay()
        torch.cuda.synchronize()
        oracle_lib.adamw8(op, specs, p_h, gh, h["mc"], h["vc"], h["ms"], h["vs"], h["m32"],
                          h["v32"], lr=hp["lr"], beta1=hp["betas"][0], beta2=hp["betas"][1],
                          eps=hp["eps"], weight_decay=hp["weight_decay"], step=4,
                          max_norm=1e-3, total_norm=tot32, nonfinite=0)
        assert_bits_equal(f32(p), p_h, f"8-bit AdamW parameters, replay {r}")
        for k, name in keys.items():
            got = st[name].cpu().numpy()[:h[k].size]
            assert_bits_equal(got, h[k], f"8-bit AdamW {name}, replay {r}")
        want_mats = [np.zeros(s.numel, np.float32) for s in specs]
        oracle_lib.gather(op, [p_h[B[k]:B[k + 1]] for k in range(m)], want_mats)
        for t in range(len(specs)):
            assert_bits_equal(f32(mats[t]), want_mats[t], f"gather tensor {t}, replay {r}")
        oracle_lib.scatter(op, want_mats, [back_h[B[k]:B[k + 1]] for k in range(m)])
        assert_bits_equal(f32(back), back_h, f"scatter, replay {r}")
    from fsdp_infra_gb300 import dbuf
    assert dbuf.dbuf_device_status(db.handle) == 0
    db.close()
