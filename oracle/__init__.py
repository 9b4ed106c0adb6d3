"""CPU oracle for the DBuffer group operators -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (``fsdp_infra_gb300``) never calls it and fails
loudly when its own CUDA library is missing.

This module is a thin ctypes wrapper over ``dbuf_oracle.c`` (plain single-threaded
C, IEEE fp32 arithmetic without contraction, fp64 sums for norms).  Arrays are
numpy arrays on the host.  Every function cites, in the C source, the passage of
the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dbuf_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")

F32, BF16 = 0, 1
QNONE, QE4M3, QINT8 = 0, 1, 2
_QUANT = {None: QNONE, "e4m3": QE4M3, "int8": QINT8}

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        L.orc_plan.argtypes = [i32, P, P, P, i32, P, i64, P, P, P]
        L.orc_plan.restype = ctypes.c_int
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.orc_f32_to_e4m3.restype = ctypes.c_uint8
        L.orc_f32_to_int8.argtypes = [ctypes.c_float]
        L.orc_f32_to_int8.restype = ctypes.c_int8
        for f in ("orc_f32_to_bf16_array", "orc_f32_to_e4m3_array", "orc_f32_to_int8_array"):
            getattr(L, f).argtypes = [P, P, i64]
            getattr(L, f).restype = None
        L.orc_pack.argtypes = [i32, P, P, P, i32, P, i32]
        L.orc_pack.restype = None
        L.orc_unpack.argtypes = [i32, P, P, P, i32, P, i32]
        L.orc_unpack.restype = None
        L.orc_scale_accum_zero.argtypes = [i32, P, P, P, i32, P, ctypes.c_float]
        L.orc_scale_accum_zero.restype = None
        L.orc_norm_nonfinite.argtypes = [i32, P, P, P, i32, P, P, P]
        L.orc_norm_nonfinite.restype = None
        L.orc_block_quant.argtypes = [i32, P, P, P, P, P, P, P, P, P]
        L.orc_block_quant.restype = i64
        L.orc_scale_offsets.argtypes = [i32, P, P, P, P, P, P]
        L.orc_scale_offsets.restype = i64
        f = ctypes.c_float
        L.orc_clip_coef.argtypes = [f, f]
        L.orc_clip_coef.restype = f
        L.orc_bias_correction.argtypes = [f, i64]
        L.orc_bias_correction.restype = f
        L.orc_adamw.argtypes = [i32, P, P, P, P, P, P, f, f, f, f, f, i64, f, f, i32]
        L.orc_adamw.restype = None
        L.orc_v_code.argtypes = [f, f]
        L.orc_v_code.restype = ctypes.c_uint8
        L.orc_state_offsets.argtypes = [i32, P, P, P]
        L.orc_state_offsets.restype = ctypes.c_int64
        L.orc_adamw8.argtypes = [i32, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                 f, f, f, f, f, i64, f, f, i32]
        L.orc_adamw8.restype = None
        for fn in ("orc_gather", "orc_scatter"):
            getattr(L, fn).argtypes = [i32, P, P, i32, P, P, i32, P]
            getattr(L, fn).restype = None
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i64(xs) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(xs, dtype=np.int64))


def _i32(xs) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(xs, dtype=np.int32))


class Plan:
    """Result of the oracle planner: S, offsets l_t, shard bounds B_k."""

    def __init__(self, S, offsets, bounds, numel):
        self.S = int(S)
        self.offsets = offsets
        self.bounds = bounds
        self.numel = numel
        self.total = int(bounds[-1])

    def __repr__(self):
        return f"OraclePlan(S={self.S}, total={self.total}, n={len(self.offsets)})"


def plan(rows: Sequence[int], cols: Sequence[int], gran_rows: Sequence[int], m: int,
         local_units: Optional[Sequence[int]] = None, align: int = 16) -> Plan:
    n = len(rows)
    r, c, g = _i64(rows), _i64(cols), _i64(gran_rows)
    units = _i32(local_units) if local_units is not None else None
    S = np.zeros(1, np.int64)
    off = np.zeros(max(n, 1), np.int64)
    bounds = np.zeros(m + 1, np.int64)
    rc = lib().orc_plan(n, _p(r), _p(c), _p(g), m, _p(units) if units is not None else None,
                        align, _p(S), _p(off), _p(bounds))
    if rc != 0:
        raise ValueError("oracle planner rejected the input")
    return Plan(S[0], off[:n].copy(), bounds, (r * c))


def plan_specs(specs, m, local_units=None, align=16) -> Plan:
    """Plan a list of workloads.TensorSpec."""
    return plan([s.rows for s in specs], [s.cols for s in specs],
                [s.gran_rows for s in specs], m, local_units, align)


def scale_offsets(specs):
    n = len(specs)
    r = _i64([s.rows for s in specs]); c = _i64([s.cols for s in specs])
    qr = _i64([s.qblock[0] for s in specs]); qc = _i64([s.qblock[1] for s in specs])
    q = _i32([_QUANT[s.quant] for s in specs])
    out = np.zeros(max(n, 1), np.int64)
    total = lib().orc_scale_offsets(n, _p(r), _p(c), _p(qr), _p(qc), _p(q), _p(out))
    return out[:n].copy(), int(total)


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_array(_p(x), _p(y), x.size)
    return y


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint8)
    lib().orc_f32_to_e4m3_array(_p(x), _p(y), x.size)
    return y


def f32_to_int8(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.int8)
    lib().orc_f32_to_int8_array(_p(x), _p(y), x.size)
    return y


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


# ----------------------------------------------------------------------------
# group operators on a flat host buffer
# ----------------------------------------------------------------------------

def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16   # bf16 bit patterns
    raise TypeError(f"oracle buffers are float32 or uint16 (bf16 bits), got {a.dtype}")


def pack(p: Plan, srcs: List[np.ndarray], buf: np.ndarray) -> None:
    n = len(srcs)
    srcs = [np.ascontiguousarray(s) for s in srcs]
    ptrs = (ctypes.c_void_p * max(n, 1))(*[s.ctypes.data for s in srcs])
    sdt = _dt(srcs[0]) if n else F32
    numel = _i64([s.size for s in srcs])
    lib().orc_pack(n, _p(p.offsets), _p(numel), ptrs, sdt, _p(buf), _dt(buf))


def unpack(p: Plan, buf: np.ndarray, dsts: List[np.ndarray]) -> None:
    n = len(dsts)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[d.ctypes.data for d in dsts])
    ddt = _dt(dsts[0]) if n else F32
    numel = _i64([d.size for d in dsts])
    lib().orc_unpack(n, _p(p.offsets), _p(numel), _p(buf), _dt(buf), ptrs, ddt)


def scale_accum_zero(p: Plan, grad: np.ndarray, acc: np.ndarray, scale: float) -> None:
    assert acc.dtype == np.float32
    lib().orc_scale_accum_zero(len(p.offsets), _p(p.offsets), _p(_i64(p.numel)), _p(grad),
                               _dt(grad), _p(acc), scale)


def norm_nonfinite(p: Plan, buf: np.ndarray):
    n = len(p.offsets)
    norms = np.zeros(max(n, 1), np.float64)
    total = np.zeros(1, np.float64)
    flag = np.zeros(1, np.int32)
    lib().orc_norm_nonfinite(n, _p(p.offsets), _p(_i64(p.numel)), _p(buf), _dt(buf),
                             _p(norms), _p(total), _p(flag))
    return norms[:n].copy(), float(total[0]), int(flag[0])


def block_quant(p: Plan, specs, buf: np.ndarray, codes: np.ndarray):
    """Returns the scales array (fp32), tensors in order, blocks row-major."""
    n = len(specs)
    r = _i64([s.rows for s in specs]); c = _i64([s.cols for s in specs])
    qr = _i64([s.qblock[0] for s in specs]); qc = _i64([s.qblock[1] for s in specs])
    q = _i32([_QUANT[s.quant] for s in specs])
    _, total = scale_offsets(specs)
    scales = np.zeros(max(total, 1), np.float32)
    assert buf.dtype == np.float32 and codes.dtype == np.uint8
    got = lib().orc_block_quant(n, _p(p.offsets), _p(r), _p(c), _p(qr), _p(qc), _p(q),
                                _p(buf), _p(codes), _p(scales))
    assert got == total
    return scales[:total].copy()


# ----------------------------------------------------------------------------
# fused group optimizer step
# ----------------------------------------------------------------------------

def clip_coef(max_norm: float, total_norm: float) -> float:
    return float(lib().orc_clip_coef(max_norm, total_norm))


def bias_correction(beta: float, step: int) -> float:
    """1 - beta^step as the optimizer steps use it (fp64 power of the fp32 beta,
    rounded to fp32)."""
    return float(lib().orc_bias_correction(beta, int(step)))


def adamw(p: Plan, params: np.ndarray, grad: np.ndarray, m: np.ndarray, v: np.ndarray, *,
          lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
          step: int, max_norm: float = 0.0, total_norm: float = 0.0,
          nonfinite: int = 0) -> None:
    """One AdamW step (step t >= 1) over the tensor ranges (in place on params, m, v)."""
    for a in (params, grad, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().orc_adamw(len(p.offsets), _p(p.offsets), _p(_i64(p.numel)), _p(params), _p(grad),
                    _p(m), _p(v), lr, beta1, beta2, eps, weight_decay, int(step), max_norm,
                    total_norm, int(nonfinite))



def v_code(v: float, scale: float) -> int:
    """The second moment's 8-bit code: nearest level (c + 1) * scale."""
    return int(lib().orc_v_code(float(v), float(scale)))


def state_offsets(specs):
    """(state_offsets[n], n_state): where each unquantised tensor's fp32 moments
    start in the compact 8-bit-AdamW state (-1 for quantised tensors)."""
    n = len(specs)
    numel = _i64([s.numel for s in specs])
    q = _i32([_QUANT[s.quant] for s in specs])
    out = np.zeros(max(n, 1), np.int64)
    total = lib().orc_state_offsets(n, _p(numel), _p(q), _p(out))
    return out[:n].copy(), int(total)


def adamw8(p: Plan, specs, params: np.ndarray, grad: np.ndarray, m_codes: np.ndarray,
           v_codes: np.ndarray, m_scales: np.ndarray, v_scales: np.ndarray, m32: np.ndarray,
           v32: np.ndarray, *, lr: float, beta1: float, beta2: float, eps: float,
           weight_decay: float, step: int, max_norm: float = 0.0,
           total_norm: float = 0.0, nonfinite: int = 0) -> None:
    """One 8-bit AdamW step (in place): INT8 block moments (codes in the flat
    buffer's layout, one fp32 scale per block) for quantised tensors, compact
    fp32 moments (m32, v32 at state_offsets) for the rest."""
    n = len(specs)
    r = _i64([s.rows for s in specs]); c = _i64([s.cols for s in specs])
    qr = _i64([s.qblock[0] for s in specs]); qc = _i64([s.qblock[1] for s in specs])
    q = _i32([_QUANT[s.quant] for s in specs])
    so, n_state = state_offsets(specs)
    so = np.ascontiguousarray(so if n else np.zeros(1, np.int64))
    for a in (params, grad, m_scales, v_scales, m32, v32):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    assert m_codes.dtype == np.uint8 and v_codes.dtype == np.uint8
    assert m32.size >= n_state and v32.size >= n_state
    assert m_codes.size >= p.total and v_codes.size >= p.total and params.size >= p.total
    lib().orc_adamw8(n, _p(p.offsets), _p(r), _p(c), _p(qr), _p(qc), _p(q), _p(so), _p(params),
                     _p(grad), _p(m_codes), _p(v_codes), _p(m_scales), _p(v_scales), _p(m32),
                     _p(v32), lr, beta1, beta2, eps, weight_decay, int(step), max_norm,
                     total_norm, int(nonfinite))


# ----------------------------------------------------------------------------
# placement orders
# ----------------------------------------------------------------------------

def shard_unit(spec) -> int:
    """g_t: elements of one shard unit (whole tensor when gran_rows is 0 or
    covers every row), at least 1."""
    numel = spec.rows * spec.cols
    g = numel if (spec.gran_rows <= 0 or spec.gran_rows >= spec.rows) else spec.gran_rows * spec.cols
    return max(g, 1)


def order(specs, kind: str = "default") -> List[int]:
    """The tensor orders the planner was studied with [veScale-FSDP, §5 Planning
    algorithm: default order, block-size order, tensor-shape order].  Read as
    stable sorts, largest first: block size = g_t, shape = (rows, cols)."""
    idx = list(range(len(specs)))
    if kind == "default":
        return idx
    if kind == "block":
        return sorted(idx, key=lambda t: -shard_unit(specs[t]))
    if kind == "shape":
        return sorted(idx, key=lambda t: (-specs[t].rows, -specs[t].cols))
    raise ValueError(kind)


# ----------------------------------------------------------------------------
# whole-matrix gather / scatter (Muon-style updates)
# ----------------------------------------------------------------------------

def _ptr_array(arrs):
    return (ctypes.c_void_p * max(len(arrs), 1))(
        *[(a.ctypes.data if a is not None else None) for a in arrs])


def gather(p: Plan, shards: List[np.ndarray], dsts: List[Optional[np.ndarray]]) -> None:
    """dsts[t] <- tensor t assembled from the m shard buffers (None = skip)."""
    dt = _dt(shards[0])
    assert len(shards) == len(p.bounds) - 1
    lib().orc_gather(len(p.offsets), _p(p.offsets), _p(_i64(p.numel)), len(shards),
                     _p(p.bounds), _ptr_array(shards), dt, _ptr_array(dsts))


def scatter(p: Plan, srcs: List[Optional[np.ndarray]], shards: List[np.ndarray]) -> None:
    """Tensor t's elements from srcs[t] back into the m shard buffers (None = skip)."""
    dt = _dt(shards[0])
    lib().orc_scatter(len(p.offsets), _p(p.offsets), _p(_i64(p.numel)), len(shards),
                      _p(p.bounds), _ptr_array(srcs), dt, _ptr_array(shards))
