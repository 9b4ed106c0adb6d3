"""Thin ctypes binding of libdbuf (include/dbuf.h): same names, argument
marshalling only.  Every computation happens in the library (host planner and
CUDA kernels); device memory and streams come from the caller (PyTorch in the
tests and the benchmark) as plain integer addresses.

There is no fallback: if libdbuf.so is missing this module raises on load.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libdbuf.so")

DBUF_OK = 0
DBUF_EINVAL = -1
DBUF_ENOMEM = -2
DBUF_ECUDA = -3
DBUF_ENOTUPLOADED = -4
DBUF_ETIMEOUT = -5
DBUF_EDEVICE = -6
DBUF_ERANGE = -7

DBUF_F32 = 0
DBUF_BF16 = 1

DBUF_QUANT_NONE = 0
DBUF_QUANT_E4M3 = 1
DBUF_QUANT_INT8 = 2

DBUF_OP_PACK = 0
DBUF_OP_UNPACK = 1
DBUF_OP_SCALE_ACCUM_ZERO = 2
DBUF_OP_NORM_NONFINITE = 3
DBUF_OP_BLOCK_QUANT = 4
DBUF_OP_ADAMW = 5

_QUANT = {None: DBUF_QUANT_NONE, "none": DBUF_QUANT_NONE, "e4m3": DBUF_QUANT_E4M3,
          "int8": DBUF_QUANT_INT8}

# Every symbol include/dbuf.h declares.
EXPORTS = ("dbuf_plan", "dbuf_plan_query", "dbuf_plan_upload", "dbuf_plan_free",
           "dbuf_pack_cast", "dbuf_unpack", "dbuf_scale_accum_zero", "dbuf_workspace_bytes",
           "dbuf_norm_nonfinite", "dbuf_norm_nonfinite_noalloc", "dbuf_block_quant",
           "dbuf_device_status", "dbuf_adamw_step", "dbuf_plan_state_offsets",
           "dbuf_adamw8_step", "dbuf_order", "dbuf_gather", "dbuf_scatter",
           "dbuf_selftest_wait_timeout", "dbuf_strerror", "dbuf_last_cuda_error",
           "dbuf_plan_slice", "dbuf_plan_slice_info", "dbuf_norm_sumsq", "dbuf_norm_finish")

# Bytes of the library's static scratch used by dbuf_norm_nonfinite_noalloc.
DBUF_NOALLOC_SCRATCH_BYTES = 1 << 20


class DbufError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {code} ({_lib_handle().dbuf_strerror(code).decode()})"
        if code == DBUF_ECUDA:
            msg += f", cudaError {_lib_handle().dbuf_last_cuda_error()}"
        super().__init__(msg)


class dbuf_adamw_hparams(ctypes.Structure):
    _fields_ = [(name, ctypes.c_float) for name in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "max_norm")] + \
               [("step", ctypes.c_int64)]


class dbuf_tensor_spec(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("gran_rows", ctypes.c_int64), ("qblock_rows", ctypes.c_int32),
                ("qblock_cols", ctypes.c_int32), ("quant", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None


def _lib_handle():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libdbuf.so is not built ({LIB_PATH}); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        try:
            import torch  # noqa: F401  (loads the shared CUDA runtime first)
        except ImportError:
            pass
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.dbuf_plan.argtypes = [P, i32, i32, P, i64, ctypes.POINTER(ctypes.c_void_p)]
        L.dbuf_plan.restype = ctypes.c_int
        L.dbuf_plan_query.argtypes = [P, P, P, P, P, P, P]
        L.dbuf_plan_query.restype = ctypes.c_int
        L.dbuf_plan_upload.argtypes = [P, P]
        L.dbuf_plan_upload.restype = ctypes.c_int
        L.dbuf_plan_free.argtypes = [P]
        L.dbuf_plan_free.restype = None
        L.dbuf_pack_cast.argtypes = [P, P, i32, P, i32, P]
        L.dbuf_pack_cast.restype = ctypes.c_int
        L.dbuf_unpack.argtypes = [P, P, i32, P, i32, P]
        L.dbuf_unpack.restype = ctypes.c_int
        L.dbuf_scale_accum_zero.argtypes = [P, P, i32, P, ctypes.c_float, P]
        L.dbuf_scale_accum_zero.restype = ctypes.c_int
        L.dbuf_workspace_bytes.argtypes = [P, i32]
        L.dbuf_workspace_bytes.restype = ctypes.c_size_t
        L.dbuf_norm_nonfinite.argtypes = [P, P, i32, P, P, P, P, ctypes.c_size_t, P]
        L.dbuf_norm_nonfinite.restype = ctypes.c_int
        L.dbuf_norm_nonfinite_noalloc.argtypes = [P, P, i32, P, P, P, P]
        L.dbuf_norm_nonfinite_noalloc.restype = ctypes.c_int
        L.dbuf_plan_slice.argtypes = [P, i32, ctypes.POINTER(ctypes.c_void_p)]
        L.dbuf_plan_slice.restype = ctypes.c_int
        L.dbuf_plan_slice_info.argtypes = [P, P, P, P, P, P]
        L.dbuf_plan_slice_info.restype = ctypes.c_int
        L.dbuf_norm_sumsq.argtypes = [P, P, i32, P, P, P, ctypes.c_size_t, P]
        L.dbuf_norm_sumsq.restype = ctypes.c_int
        L.dbuf_norm_finish.argtypes = [P, P, P, P, P]
        L.dbuf_norm_finish.restype = ctypes.c_int
        L.dbuf_block_quant.argtypes = [P, P, P, P, P]
        L.dbuf_block_quant.restype = ctypes.c_int
        L.dbuf_adamw_step.argtypes = [P, P, P, P, P, P, P, P, P]
        L.dbuf_adamw_step.restype = ctypes.c_int
        L.dbuf_plan_state_offsets.argtypes = [P, P, P]
        L.dbuf_plan_state_offsets.restype = ctypes.c_int
        L.dbuf_adamw8_step.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P]
        L.dbuf_adamw8_step.restype = ctypes.c_int
        L.dbuf_order.argtypes = [P, i32, i32, P]
        L.dbuf_order.restype = ctypes.c_int
        L.dbuf_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
        L.dbuf_selftest_wait_timeout.restype = ctypes.c_int
        for fn in ("dbuf_gather", "dbuf_scatter"):
            getattr(L, fn).argtypes = [P, P, i32, P, P]
            getattr(L, fn).restype = ctypes.c_int
        L.dbuf_device_status.argtypes = [P, P, P]
        L.dbuf_device_status.restype = ctypes.c_int
        L.dbuf_strerror.argtypes = [ctypes.c_int]
        L.dbuf_strerror.restype = ctypes.c_char_p
        L.dbuf_last_cuda_error.argtypes = []
        L.dbuf_last_cuda_error.restype = ctypes.c_int
        _lib = L
    return _lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _lib_handle()


def _check(rc: int, where: str) -> None:
    if rc != DBUF_OK:
        raise DbufError(rc, where)


def _spec_array(specs) -> ctypes.Array:
    arr = (dbuf_tensor_spec * max(len(specs), 1))()
    for i, s in enumerate(specs):
        if isinstance(s, (tuple, list)):
            rows, cols, gran = s[0], s[1], s[2]
            qb = s[3] if len(s) > 3 else (0, 0)
            q = s[4] if len(s) > 4 else None
        else:
            rows, cols, gran = s.rows, s.cols, s.gran_rows
            qb, q = getattr(s, "qblock", (0, 0)), getattr(s, "quant", None)
        arr[i] = dbuf_tensor_spec(rows, cols, gran, qb[0], qb[1], _QUANT.get(q, q), 0)
    return arr


def dbuf_plan(specs: Sequence, m: int, local_units: Optional[Sequence[int]] = None,
              align_elems: int = 16) -> int:
    """Plan a tensor group; returns the opaque plan handle (an int)."""
    arr = _spec_array(specs)
    units = (ctypes.c_int32 * m)(*local_units) if local_units is not None else None
    out = ctypes.c_void_p()
    _check(_lib_handle().dbuf_plan(arr, len(specs), m, units, align_elems, ctypes.byref(out)),
           "dbuf_plan")
    return out.value


DBUF_ORDER = {"default": 0, "block": 1, "shape": 2}


def dbuf_order(specs, kind: str = "default") -> list:
    """Placement permutation of the specs for one of the studied orders:
    perm[i] is the index of the tensor placed i-th."""
    arr = _spec_array(specs)
    perm = (ctypes.c_int32 * max(len(specs), 1))()
    _check(_lib_handle().dbuf_order(arr, len(specs), DBUF_ORDER[kind], perm), "dbuf_order")
    return list(perm)[:len(specs)]


def dbuf_plan_query(plan: int, n: int, m: int) -> dict:
    S, total, ns = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    off = (ctypes.c_int64 * max(n, 1))()
    bounds = (ctypes.c_int64 * (m + 1))()
    soff = (ctypes.c_int64 * max(n, 1))()
    _check(_lib_handle().dbuf_plan_query(plan, ctypes.byref(S), ctypes.byref(total), off, bounds,
                                         soff, ctypes.byref(ns)), "dbuf_plan_query")
    return {"S": S.value, "total": total.value, "offsets": list(off)[:n],
            "shard_bounds": list(bounds), "scale_offsets": list(soff)[:n], "n_scales": ns.value}


def dbuf_plan_slice(plan: int, k: int) -> int:
    """The plan of shard slice k as a rank's local buffer (a new plan handle)."""
    out = ctypes.c_void_p()
    _check(_lib_handle().dbuf_plan_slice(plan, k, ctypes.byref(out)), "dbuf_plan_slice")
    return out.value


def dbuf_plan_slice_info(slice_plan: int, n: int) -> dict:
    k, off, base = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    src = (ctypes.c_int64 * max(n, 1))()
    num = (ctypes.c_int64 * max(n, 1))()
    _check(_lib_handle().dbuf_plan_slice_info(slice_plan, ctypes.byref(k), ctypes.byref(off), src,
                                              num, ctypes.byref(base)), "dbuf_plan_slice_info")
    return {"k": k.value, "global_offset": off.value, "src_offsets": list(src)[:n],
            "numels": list(num)[:n], "scale_base": base.value}


def dbuf_norm_sumsq(plan: int, buf: int, dtype: int, tensor_sumsq: int, nonfinite: int,
                    workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _check(_lib_handle().dbuf_norm_sumsq(plan, buf, dtype, tensor_sumsq, nonfinite, workspace,
                                         workspace_bytes, stream), "dbuf_norm_sumsq")


def dbuf_norm_finish(plan: int, tensor_sumsq: int, tensor_norms: int, total_norm: int,
                     stream: int = 0) -> None:
    _check(_lib_handle().dbuf_norm_finish(plan, tensor_sumsq, tensor_norms, total_norm, stream),
           "dbuf_norm_finish")


def dbuf_plan_upload(plan: int, stream: int = 0) -> None:
    _check(_lib_handle().dbuf_plan_upload(plan, stream), "dbuf_plan_upload")


def dbuf_plan_free(plan: int) -> None:
    _lib_handle().dbuf_plan_free(plan)


def dbuf_pack_cast(plan: int, src_ptrs: int, src_dtype: int, buf: int, buf_dtype: int,
                   stream: int = 0) -> None:
    _check(_lib_handle().dbuf_pack_cast(plan, src_ptrs, src_dtype, buf, buf_dtype, stream),
           "dbuf_pack_cast")


def dbuf_unpack(plan: int, buf: int, buf_dtype: int, dst_ptrs: int, dst_dtype: int,
                stream: int = 0) -> None:
    _check(_lib_handle().dbuf_unpack(plan, buf, buf_dtype, dst_ptrs, dst_dtype, stream),
           "dbuf_unpack")


def dbuf_scale_accum_zero(plan: int, grad: int, grad_dtype: int, acc: int, scale: float,
                          stream: int = 0) -> None:
    _check(_lib_handle().dbuf_scale_accum_zero(plan, grad, grad_dtype, acc, scale, stream),
           "dbuf_scale_accum_zero")


def dbuf_workspace_bytes(plan: int, op: int) -> int:
    return int(_lib_handle().dbuf_workspace_bytes(plan, op))


def dbuf_norm_nonfinite(plan: int, buf: int, dtype: int, tensor_norms: int, total_norm: int,
                        nonfinite: int, workspace: int, workspace_bytes: int,
                        stream: int = 0) -> None:
    _check(_lib_handle().dbuf_norm_nonfinite(plan, buf, dtype, tensor_norms, total_norm,
                                             nonfinite, workspace, workspace_bytes, stream),
           "dbuf_norm_nonfinite")


def dbuf_norm_nonfinite_noalloc(plan: int, buf: int, dtype: int, tensor_norms: int,
                                total_norm: int, nonfinite: int, stream: int = 0) -> None:
    """dbuf_norm_nonfinite without a workspace, for callers that cannot allocate
    device memory: the library's static scratch is used instead (see dbuf.h)."""
    _check(_lib_handle().dbuf_norm_nonfinite_noalloc(plan, buf, dtype, tensor_norms, total_norm,
                                                     nonfinite, stream),
           "dbuf_norm_nonfinite_noalloc")


def dbuf_block_quant(plan: int, buf: int, codes: int, scales: int, stream: int = 0) -> None:
    _check(_lib_handle().dbuf_block_quant(plan, buf, codes, scales, stream), "dbuf_block_quant")


def dbuf_adamw_step(plan: int, params: int, grads: int, exp_avg: int, exp_avg_sq: int, *,
                    step: int, lr: float, beta1: float, beta2: float, eps: float,
                    weight_decay: float, max_norm: float = 0.0, total_norm: int = 0,
                    nonfinite: int = 0, stream: int = 0) -> None:
    """One AdamW step (step >= 1) over the tensor ranges; total_norm / nonfinite
    are optional device pointers (0 = not given)."""
    hp = dbuf_adamw_hparams(lr, beta1, beta2, eps, weight_decay, max_norm, step)
    _check(_lib_handle().dbuf_adamw_step(plan, params, grads, exp_avg, exp_avg_sq,
                                         ctypes.byref(hp), total_norm or None, nonfinite or None,
                                         stream), "dbuf_adamw_step")


def dbuf_plan_state_offsets(plan: int, n: int):
    """(state_offsets[n], n_state) of the compact fp32 moments of the 8-bit step."""
    off = (ctypes.c_int64 * max(n, 1))()
    ns = ctypes.c_int64()
    _check(_lib_handle().dbuf_plan_state_offsets(plan, off, ctypes.byref(ns)),
           "dbuf_plan_state_offsets")
    return list(off)[:n], ns.value


def dbuf_adamw8_step(plan: int, params: int, grads: int, exp_avg_codes: int,
                     exp_avg_sq_codes: int, exp_avg_scales: int, exp_avg_sq_scales: int,
                     exp_avg_fp32: int, exp_avg_sq_fp32: int, *, step: int, lr: float,
                     beta1: float, beta2: float, eps: float, weight_decay: float,
                     max_norm: float = 0.0, total_norm: int = 0, nonfinite: int = 0,
                     stream: int = 0) -> None:
    """One 8-bit AdamW step (step >= 1, block-quantised moments); pointers as in
    dbuf.h, 0 for the optional ones."""
    hp = dbuf_adamw_hparams(lr, beta1, beta2, eps, weight_decay, max_norm, step)
    _check(_lib_handle().dbuf_adamw8_step(plan, params, grads, exp_avg_codes or None,
                                          exp_avg_sq_codes or None, exp_avg_scales or None,
                                          exp_avg_sq_scales or None, exp_avg_fp32 or None,
                                          exp_avg_sq_fp32 or None, ctypes.byref(hp),
                                          total_norm or None, nonfinite or None, stream),
           "dbuf_adamw8_step")


def dbuf_gather(plan: int, shard_ptrs: int, dtype: int, dst_ptrs: int, stream: int = 0) -> None:
    _check(_lib_handle().dbuf_gather(plan, shard_ptrs, dtype, dst_ptrs, stream), "dbuf_gather")


def dbuf_scatter(plan: int, src_ptrs: int, dtype: int, shard_ptrs: int, stream: int = 0) -> None:
    _check(_lib_handle().dbuf_scatter(plan, src_ptrs, dtype, shard_ptrs, stream), "dbuf_scatter")


def dbuf_selftest_wait_timeout(plan: int, tries: int, stream: int = 0) -> None:
    """Diagnostic: a device wait that runs out and records DBUF_ETIMEOUT."""
    _check(_lib_handle().dbuf_selftest_wait_timeout(plan, tries, stream),
           "dbuf_selftest_wait_timeout")


def dbuf_device_status(plan: int, stream: int = 0) -> int:
    """Reads and clears the plan's device status word (0 or DBUF_ETIMEOUT)."""
    v = ctypes.c_int32()
    _check(_lib_handle().dbuf_device_status(plan, ctypes.byref(v), stream), "dbuf_device_status")
    return v.value


def dbuf_strerror(code: int) -> str:
    return _lib_handle().dbuf_strerror(code).decode()


def dbuf_last_cuda_error() -> int:
    return int(_lib_handle().dbuf_last_cuda_error())
