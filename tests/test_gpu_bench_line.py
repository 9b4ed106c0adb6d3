"""bench.py on the GPU prints one JSON line with the benchmark's fields: the
job throughput, the roofline object of the dominant kernel, the CPU-oracle
baseline, the end-to-end figure with the bytes it copies, the launch count and
the SM clocks sampled during the timed region.  The tiny two-layer group keeps
the run to seconds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_fields(dbuf_lib, oracle_lib):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                        "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])

    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["dtype"] == "f32" and d["vs_baseline"] is None
    assert d["config"]["key"] == "tiny" and d["config"]["workload"]

    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    # the recorded DRAM traffic belongs to the 7B-layer launch, not to this workload
    assert roof["traffic"] is None

    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0

    # 5 step operators on the tiny group's one DBuffer (6 launches: the norm has a
    # finishing launch), every step
    assert d["gpu_launches"] == 6 * d["steps"]

    # a timed region of microseconds may fall between two nvidia-smi samples
    clocks = d["clocks"]
    assert isinstance(clocks["reasons"], list)
    if clocks.get("samples"):
        assert clocks["sm_max_mhz"] > 0 and clocks["sm_mhz"] > 0
    else:
        assert clocks["reasons"]
    for op in ("pack_cast", "unpack", "scale_accum_zero", "norm_nonfinite", "block_quant"):
        assert d["ops"][op]["gbs"] > 0


@pytest.mark.gpu
def test_bench_exchange_mode_on_one_gpu(dbuf_lib):
    """--exchange runs the sharded step (ShardedStep around NCCL collectives) with
    m = the number of GPUs; on one GPU the process group has one rank, which
    exercises the whole code path (plans, slice plans, collectives, operators)."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--exchange",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["mode"] == "exchange" and d["n_gpus"] == 1 and d["config"]["m"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["collective_bytes_per_rank"] > 0 and d["op_bytes_per_rank"] > 0
