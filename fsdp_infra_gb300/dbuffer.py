"""DBuffer: a planned flat buffer for one tensor group, on top of the C ABI.

PyTorch provides device memory and streams only; every step of the group
operators runs in libdbuf's kernels through the binding in ``dbuf.py``.  This
class keeps a plan handle and the device-side pointer tables of the user
tensors, and exposes zero-copy views of each tensor inside a buffer
("veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer:
zero-copy access through a persistent address mapping).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import dbuf as _c

_DT = {torch.float32: _c.DBUF_F32, torch.bfloat16: _c.DBUF_BF16}


def dtype_code(t: torch.dtype) -> int:
    try:
        return _DT[t]
    except KeyError:
        raise TypeError(f"DBuffer buffers are float32 or bfloat16, not {t}") from None


class DBuffer:
    """One planned tensor group: layout, descriptor tables on the device, and
    the group operators over buffers of that layout."""

    def __init__(self, specs: Sequence, m: int, local_units: Optional[Sequence[int]] = None,
                 align_elems: int = 16, device: Optional[torch.device] = None):
        self.specs = list(specs)
        self.n = len(self.specs)
        self.local_units = list(local_units) if local_units is not None else None
        self._setup(_c.dbuf_plan(self.specs, m, local_units, align_elems), m, device)
        self.slice_k = None

    def _setup(self, handle: int, m: int, device) -> None:
        self.m = m
        self.handle = handle
        q = _c.dbuf_plan_query(self.handle, self.n, m)
        self.S: int = q["S"]
        self.total: int = q["total"]
        self.offsets: List[int] = q["offsets"]
        self.shard_bounds: List[int] = q["shard_bounds"]
        self.scale_offsets: List[int] = q["scale_offsets"]
        self.n_scales: int = q["n_scales"]
        self.state_offsets, self.n_state = _c.dbuf_plan_state_offsets(self.handle, self.n)
        self.numel = [int(s.rows) * int(s.cols) if not isinstance(s, (tuple, list))
                      else int(s[0]) * int(s[1]) for s in self.specs]
        dev = torch.device(device if device is not None else "cuda")
        if dev.type == "cuda" and dev.index is None and torch.cuda.is_available():
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self._ptr_tables: Dict[Tuple[int, ...], torch.Tensor] = {}
        self._workspace: Optional[torch.Tensor] = None
        self.uploaded = False

    def slice(self, k: int) -> "DBuffer":
        """Shard slice k as a rank's local DBuffer (not yet uploaded): its buffers
        hold the B_{k+1} - B_k elements of [B_k, B_{k+1}); the group operators run
        on the tensors' pieces inside the slice and take the same whole user
        tensors as this DBuffer."""
        sl = DBuffer.__new__(DBuffer)
        sl.specs = self.specs
        sl.n = self.n
        sl.local_units = None
        sl._setup(_c.dbuf_plan_slice(self.handle, k), 1, self.device)
        info = _c.dbuf_plan_slice_info(sl.handle, sl.n)
        sl.slice_k = info["k"]
        sl.global_offset = info["global_offset"]
        sl.src_offsets = info["src_offsets"]
        sl.piece_numels = info["numels"]
        sl.scale_base = info["scale_base"]
        return sl

    # -- lifetime ------------------------------------------------------------
    def upload(self, stream: Optional[torch.cuda.Stream] = None) -> "DBuffer":
        with torch.cuda.device(self.device):
            st = stream if stream is not None else torch.cuda.current_stream()
            _c.dbuf_plan_upload(self.handle, st.cuda_stream)
        self.uploaded = True
        return self

    def close(self) -> None:
        if self.handle:
            _c.dbuf_plan_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- memory helpers (allocation only) -------------------------------------
    def new_buffer(self, dtype: torch.dtype, zero: bool = True) -> torch.Tensor:
        """A flat buffer of `total` elements; padding starts (and stays) zero."""
        f = torch.zeros if zero else torch.empty
        return f(self.total, dtype=dtype, device=self.device)

    def view(self, buf: torch.Tensor, t: int) -> torch.Tensor:
        """Zero-copy view of tensor t inside `buf`."""
        s = self.specs[t]
        rows, cols = (s[0], s[1]) if isinstance(s, (tuple, list)) else (s.rows, s.cols)
        o = self.offsets[t]
        return buf[o:o + rows * cols].view(rows, cols)

    def ptr_table(self, tensors: Sequence[torch.Tensor]) -> torch.Tensor:
        """Device array of the tensors' data pointers, cached per tuple of
        (pointer, element count, dtype): the checks run once per new tuple."""
        if len(tensors) != self.n:
            raise ValueError(f"expected {self.n} tensors, got {len(tensors)}")
        key = tuple((x.data_ptr(), x.numel(), x.dtype) for x in tensors)
        tab = self._ptr_tables.get(key)
        if tab is None:
            for t, x in enumerate(tensors):
                if x.dtype != tensors[0].dtype:
                    raise TypeError("all tensors of one call must share one dtype")
                if not x.is_contiguous() or x.numel() != self.numel[t]:
                    raise ValueError(f"tensor {t} must be contiguous with {self.numel[t]} elements")
                if x.device != self.device:
                    raise ValueError(f"tensor {t} is on {x.device}, expected {self.device}")
            ptrs = [k[0] for k in key] or [0]
            tab = self._settled(torch.tensor(ptrs, dtype=torch.int64, device=self.device))
            self._ptr_tables[key] = tab
        return tab

    def _settled(self, t: torch.Tensor) -> torch.Tensor:
        """A cached device tensor just written on the current stream, made complete
        before it is returned so that calls on any stream may use it (once per
        cache entry; entries are made before any stream capture)."""
        if not torch.cuda.is_current_stream_capturing():
            torch.cuda.current_stream(self.device).synchronize()
        return t

    def workspace_bytes(self) -> int:
        return _c.dbuf_workspace_bytes(self.handle, _c.DBUF_OP_NORM_NONFINITE)

    def new_workspace(self) -> torch.Tensor:
        """A norm workspace of its own, for a caller whose norm calls may overlap
        those of other streams (zero-filled: the completion counters start at
        zero and every call leaves them at zero again)."""
        return self._settled(torch.zeros(max(self.workspace_bytes(), 1), dtype=torch.uint8,
                                         device=self.device))

    def workspace(self) -> torch.Tensor:
        """The DBuffer's own norm workspace: calls that use it must not overlap on
        the GPU (one stream at a time)."""
        nbytes = self.workspace_bytes()
        if self._workspace is None or self._workspace.numel() < nbytes:
            self._workspace = self.new_workspace()
        return self._workspace

    # -- group operators ---------------------------------------------------------
    @staticmethod
    def _stream(stream):
        return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream

    def _check_buf(self, buf: torch.Tensor):
        if buf.numel() < self.total or not buf.is_contiguous() or buf.device != self.device:
            raise ValueError("buffer must be a contiguous device tensor of `total` elements")

    def pack_cast(self, srcs: Sequence[torch.Tensor], buf: torch.Tensor, stream=None) -> None:
        self._check_buf(buf)
        sdt = dtype_code(srcs[0].dtype) if srcs else _c.DBUF_F32
        tab = self.ptr_table(srcs)
        _c.dbuf_pack_cast(self.handle, tab.data_ptr(), sdt, buf.data_ptr(), dtype_code(buf.dtype),
                          self._stream(stream))

    def unpack(self, buf: torch.Tensor, dsts: Sequence[torch.Tensor], stream=None) -> None:
        self._check_buf(buf)
        ddt = dtype_code(dsts[0].dtype) if dsts else _c.DBUF_F32
        tab = self.ptr_table(dsts)
        _c.dbuf_unpack(self.handle, buf.data_ptr(), dtype_code(buf.dtype), tab.data_ptr(), ddt,
                       self._stream(stream))

    def scale_accum_zero(self, grad: torch.Tensor, acc: torch.Tensor, scale: float,
                         stream=None) -> None:
        self._check_buf(grad)
        self._check_buf(acc)
        if acc.dtype != torch.float32:
            raise TypeError("the accumulator is float32")
        _c.dbuf_scale_accum_zero(self.handle, grad.data_ptr(), dtype_code(grad.dtype),
                                 acc.data_ptr(), float(scale), self._stream(stream))

    def norm_nonfinite(self, buf: torch.Tensor, out: Optional[Tuple] = None, stream=None,
                       workspace: Optional[torch.Tensor] = None):
        """Returns device tensors (tensor_norms[n] f32, total_norm[1] f32, nonfinite[1] i32).
        `workspace` (from new_workspace) replaces the DBuffer's own for calls that may
        overlap other streams' norm calls."""
        self._check_buf(buf)
        if out is None:
            out = (torch.empty(max(self.n, 1), dtype=torch.float32, device=self.device),
                   torch.empty(1, dtype=torch.float32, device=self.device),
                   torch.empty(1, dtype=torch.int32, device=self.device))
        norms, total, flag = out
        ws = self.workspace() if workspace is None else workspace
        _c.dbuf_norm_nonfinite(self.handle, buf.data_ptr(), dtype_code(buf.dtype),
                               norms.data_ptr(), total.data_ptr(), flag.data_ptr(),
                               ws.data_ptr(), ws.numel(), self._stream(stream))
        return norms[:self.n], total, flag

    def norm_sumsq(self, buf: torch.Tensor, out: Optional[Tuple] = None, stream=None,
                   workspace: Optional[torch.Tensor] = None):
        """Per-tensor fp64 sums of squares and the non-finite flag (device tensors
        sumsq[n] f64, nonfinite[1] i32): the partials a sharded norm adds up."""
        self._check_buf(buf)
        if out is None:
            out = (torch.empty(max(self.n, 1), dtype=torch.float64, device=self.device),
                   torch.empty(1, dtype=torch.int32, device=self.device))
        sumsq, flag = out
        ws = self.workspace() if workspace is None else workspace
        _c.dbuf_norm_sumsq(self.handle, buf.data_ptr(), dtype_code(buf.dtype), sumsq.data_ptr(),
                           flag.data_ptr(), ws.data_ptr(), ws.numel(), self._stream(stream))
        return sumsq[:self.n], flag

    def norm_finish(self, sumsq: torch.Tensor, out: Optional[Tuple] = None, stream=None):
        """Norms from (all-reduced) per-tensor sums of squares: (tensor_norms[n]
        f32, total_norm[1] f32) device tensors."""
        if sumsq.dtype != torch.float64 or sumsq.numel() < self.n or sumsq.device != self.device:
            raise ValueError("sumsq must be a float64 device tensor of n elements")
        if out is None:
            out = (torch.empty(max(self.n, 1), dtype=torch.float32, device=self.device),
                   torch.empty(1, dtype=torch.float32, device=self.device))
        norms, total = out
        _c.dbuf_norm_finish(self.handle, sumsq.data_ptr(), norms.data_ptr(), total.data_ptr(),
                            self._stream(stream))
        return norms[:self.n], total

    def block_quant(self, buf: torch.Tensor, codes: Optional[torch.Tensor] = None,
                    scales: Optional[torch.Tensor] = None, stream=None):
        """Returns (codes uint8[total], scales f32[n_scales])."""
        self._check_buf(buf)
        if buf.dtype != torch.float32:
            raise TypeError("block quantisation reads a float32 buffer")
        if codes is None:
            codes = torch.zeros(self.total, dtype=torch.uint8, device=self.device)
        if scales is None:
            scales = torch.empty(max(self.n_scales, 1), dtype=torch.float32, device=self.device)
        _c.dbuf_block_quant(self.handle, buf.data_ptr(), codes.data_ptr(), scales.data_ptr(),
                            self._stream(stream))
        return codes, scales[:self.n_scales]

    def adamw_step(self, params: torch.Tensor, grads: torch.Tensor, exp_avg: torch.Tensor,
                   exp_avg_sq: torch.Tensor, *, step: int, lr: float, betas=(0.9, 0.999),
                   eps: float = 1e-8, weight_decay: float = 0.0, max_norm: float = 0.0,
                   total_norm: Optional[torch.Tensor] = None,
                   nonfinite: Optional[torch.Tensor] = None, stream=None) -> None:
        """One fused AdamW step over fp32 buffers of this layout (step >= 1; the
        library forms the bias corrections)."""
        for b in (params, grads, exp_avg, exp_avg_sq):
            self._check_buf(b)
            if b.dtype != torch.float32:
                raise TypeError("AdamW buffers are float32")
        b1, b2 = betas
        _c.dbuf_adamw_step(self.handle, params.data_ptr(), grads.data_ptr(), exp_avg.data_ptr(),
                           exp_avg_sq.data_ptr(), step=step, lr=lr, beta1=b1, beta2=b2,
                           eps=eps, weight_decay=weight_decay, max_norm=max_norm,
                           total_norm=total_norm.data_ptr() if total_norm is not None else 0,
                           nonfinite=nonfinite.data_ptr() if nonfinite is not None else 0,
                           stream=self._stream(stream))

    # -- 8-bit AdamW -----------------------------------------------------------
    def new_adamw8_state(self) -> Dict[str, torch.Tensor]:
        """Zero 8-bit AdamW state: uint8 codes of m and v in the flat buffer's
        layout, fp32 block scales, compact fp32 moments of unquantised tensors."""
        def z(n, dt):
            return torch.zeros(max(n, 1), dtype=dt, device=self.device)
        return {"m_codes": z(self.total, torch.uint8), "v_codes": z(self.total, torch.uint8),
                "m_scales": z(self.n_scales, torch.float32),
                "v_scales": z(self.n_scales, torch.float32),
                "m32": z(self.n_state, torch.float32), "v32": z(self.n_state, torch.float32)}

    def adamw8_step(self, params: torch.Tensor, grads: torch.Tensor, state: Dict[str, torch.Tensor],
                    *, step: int, lr: float, betas=(0.9, 0.999), eps: float = 1e-8,
                    weight_decay: float = 0.0, max_norm: float = 0.0,
                    total_norm: Optional[torch.Tensor] = None,
                    nonfinite: Optional[torch.Tensor] = None, stream=None) -> None:
        """One fused 8-bit AdamW step (step >= 1) on the state of new_adamw8_state."""
        for b in (params, grads):
            self._check_buf(b)
            if b.dtype != torch.float32:
                raise TypeError("AdamW parameters and gradients are float32")
        need = {"m_codes": (self.total, torch.uint8), "v_codes": (self.total, torch.uint8),
                "m_scales": (self.n_scales, torch.float32),
                "v_scales": (self.n_scales, torch.float32),
                "m32": (self.n_state, torch.float32), "v32": (self.n_state, torch.float32)}
        for k, (n, dt) in need.items():
            t = state[k]
            if t.dtype != dt or t.numel() < n or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"8-bit AdamW state {k}: want {n} {dt} on {self.device}")
        b1, b2 = betas
        _c.dbuf_adamw8_step(self.handle, params.data_ptr(), grads.data_ptr(),
                            state["m_codes"].data_ptr(), state["v_codes"].data_ptr(),
                            state["m_scales"].data_ptr(), state["v_scales"].data_ptr(),
                            state["m32"].data_ptr(), state["v32"].data_ptr(), step=step,
                            lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=weight_decay,
                            max_norm=max_norm,
                            total_norm=total_norm.data_ptr() if total_norm is not None else 0,
                            nonfinite=nonfinite.data_ptr() if nonfinite is not None else 0,
                            stream=self._stream(stream))

    # -- whole-matrix gather / scatter -------------------------------------------
    def shard_sizes(self) -> List[int]:
        """Elements of each of the m shard slices (B_{k+1} - B_k)."""
        b = self.shard_bounds
        return [b[k + 1] - b[k] for k in range(self.m)]

    def _opt_ptr_table(self, tensors, numels, what) -> torch.Tensor:
        """Device array of data pointers (0 for None), cached per tuple of
        (pointer, element count, dtype) like ptr_table."""
        key = (what,) + tuple(None if x is None else (x.data_ptr(), x.numel(), x.dtype)
                              for x in tensors)
        tab = self._ptr_tables.get(key)
        if tab is not None:
            return tab
        ptrs = []
        for t, x in enumerate(tensors):
            if x is None:
                ptrs.append(0)
                continue
            if not x.is_contiguous() or x.numel() != numels[t] or x.device != self.device:
                raise ValueError(f"{what} {t}: want a contiguous tensor of {numels[t]} "
                                 f"elements on {self.device}")
            ptrs.append(x.data_ptr())
        tab = self._settled(torch.tensor(ptrs or [0], dtype=torch.int64, device=self.device))
        self._ptr_tables[key] = tab
        return tab

    def gather(self, shards: Sequence[torch.Tensor], dsts: Sequence[Optional[torch.Tensor]],
               stream=None) -> None:
        """dsts[t] <- tensor t's full matrix assembled from the m shard buffers
        (None skips the tensor)."""
        if len(shards) != self.m or len(dsts) != self.n:
            raise ValueError("gather wants m shards and n destinations")
        dt = dtype_code(shards[0].dtype)
        if any(x is not None and x.dtype != shards[0].dtype for x in list(shards) + list(dsts)):
            raise TypeError("shards and matrices must share one dtype")
        sh = self._opt_ptr_table(shards, self.shard_sizes(), "shard")
        tab = self._opt_ptr_table(dsts, self.numel, "matrix")
        _c.dbuf_gather(self.handle, sh.data_ptr(), dt, tab.data_ptr(), self._stream(stream))

    def scatter(self, srcs: Sequence[Optional[torch.Tensor]], shards: Sequence[torch.Tensor],
                stream=None) -> None:
        """Tensor t's full matrix srcs[t] back into the m shard buffers (None skips)."""
        if len(shards) != self.m or len(srcs) != self.n:
            raise ValueError("scatter wants n sources and m shards")
        dt = dtype_code(shards[0].dtype)
        if any(x is not None and x.dtype != shards[0].dtype for x in list(shards) + list(srcs)):
            raise TypeError("shards and matrices must share one dtype")
        sh = self._opt_ptr_table(shards, self.shard_sizes(), "shard")
        tab = self._opt_ptr_table(srcs, self.numel, "matrix")
        _c.dbuf_scatter(self.handle, tab.data_ptr(), dt, sh.data_ptr(), self._stream(stream))

