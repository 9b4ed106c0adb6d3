"""The C-ABI library loads, exports every symbol include/dbuf.h declares, and
rejects bad arguments on the host before touching any GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dbuf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dbuf_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ["dbuf_plan", "dbuf_pack_cast", "dbuf_unpack", "dbuf_scale_accum_zero",
              "dbuf_norm_nonfinite", "dbuf_block_quant"]:
        assert s in syms


def test_library_exports_every_declared_symbol(dbuf_lib):
    lib = ctypes.CDLL(dbuf_lib.LIB_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing
    assert set(declared_symbols()) == set(dbuf_lib.EXPORTS)


def test_struct_layout(dbuf_lib):
    assert ctypes.sizeof(dbuf_lib.dbuf_tensor_spec) == 40


def test_plan_rejects_bad_arguments(dbuf_lib):
    d = dbuf_lib
    with pytest.raises(d.DbufError) as e:
        d.dbuf_plan([(4, 4, 1)], 0)
    assert e.value.code == d.DBUF_EINVAL
    with pytest.raises(d.DbufError):
        d.dbuf_plan([(-1, 4, 1)], 2)
    with pytest.raises(d.DbufError):
        d.dbuf_plan([(4, 4, 1)], 2, local_units=[1, 0])
    with pytest.raises(d.DbufError):
        d.dbuf_plan([(4, 4, 1)], 2, align_elems=0)
    # a quantised tensor whose shard unit would split a 128-row block
    with pytest.raises(d.DbufError):
        d.dbuf_plan([(256, 128, 64, (128, 128), "e4m3")], 2)
    with pytest.raises(d.DbufError) as e:
        d.dbuf_plan([(1 << 40, 1 << 20, 1)], 2)
    assert e.value.code == d.DBUF_ERANGE
    # one quantisation block of 2^31 elements or more
    with pytest.raises(d.DbufError) as e:
        d.dbuf_plan([(1 << 16, 1 << 15, 0, (0, 0), "int8")], 2)
    assert e.value.code == d.DBUF_ERANGE
    p = d.dbuf_plan([(1 << 16, (1 << 15) - 1, 0, (0, 0), "int8")], 2)
    d.dbuf_plan_free(p)


def test_operators_refuse_unuploaded_plan_without_gpu(dbuf_lib):
    d = dbuf_lib
    p = d.dbuf_plan([(8, 8, 1), (16, 1, 1)], 2)
    try:
        for call in [lambda: d.dbuf_pack_cast(p, 0, d.DBUF_F32, 0, d.DBUF_F32),
                     lambda: d.dbuf_unpack(p, 0, d.DBUF_F32, 0, d.DBUF_F32),
                     lambda: d.dbuf_scale_accum_zero(p, 0, d.DBUF_F32, 0, 0.5),
                     lambda: d.dbuf_norm_nonfinite(p, 0, d.DBUF_F32, 0, 0, 0, 0, 0),
                     lambda: d.dbuf_block_quant(p, 0, 0, 0),
                     lambda: d.dbuf_adamw8_step(p, 0, 0, 0, 0, 0, 0, 0, 0, step=1, lr=1e-3,
                                                beta1=0.9, beta2=0.95, eps=1e-8,
                                                weight_decay=0.0),
                     lambda: d.dbuf_gather(p, 0, d.DBUF_F32, 0),
                     lambda: d.dbuf_scatter(p, 0, d.DBUF_F32, 0),
                     lambda: d.dbuf_selftest_wait_timeout(p, 100)]:
            with pytest.raises(d.DbufError) as e:
                call()
            assert e.value.code == d.DBUF_ENOTUPLOADED
        assert d.dbuf_workspace_bytes(p, d.DBUF_OP_NORM_NONFINITE) > 0
        assert d.dbuf_workspace_bytes(p, d.DBUF_OP_PACK) == 0
    finally:
        d.dbuf_plan_free(p)
    d.dbuf_plan_free(0)   # NULL is a no-op


def test_strerror(dbuf_lib):
    d = dbuf_lib
    assert d.dbuf_strerror(0) == "ok"
    assert "not uploaded" in d.dbuf_strerror(d.DBUF_ENOTUPLOADED)
    assert d.dbuf_strerror(12345) == "unknown error"


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    import fsdp_infra_gb300.dbuf as d
    monkeypatch.setattr(d, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(d, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        d.library()


def test_adamw_rejects_bad_step_and_betas_without_gpu(dbuf_lib):
    """The library forms 1 - beta^t itself: step < 1, or a beta that makes a
    correction zero, is refused before the plan is even looked at."""
    d = dbuf_lib
    p = d.dbuf_plan([(8, 8, 1)], 2)
    try:
        kw = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
        for bad in [dict(kw, step=0), dict(kw, step=-3), dict(kw, step=1, beta1=1.0),
                    dict(kw, step=5, beta2=1.0)]:
            for call in (lambda: d.dbuf_adamw_step(p, 0, 0, 0, 0, **bad),
                         lambda: d.dbuf_adamw8_step(p, 0, 0, 0, 0, 0, 0, 0, 0, **bad)):
                with pytest.raises(d.DbufError) as e:
                    call()
                assert e.value.code == d.DBUF_EINVAL
        with pytest.raises(d.DbufError) as e:
            d.dbuf_adamw_step(p, 0, 0, 0, 0, step=1, **kw)
        assert e.value.code == d.DBUF_ENOTUPLOADED
    finally:
        d.dbuf_plan_free(p)
