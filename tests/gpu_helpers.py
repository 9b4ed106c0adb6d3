"""Helpers of the GPU parity tests: seeded inputs for a planned group, host
copies for the oracle, and comparisons.  Expected values come from the oracle
only; the CUDA path is only ever the thing being checked."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy in the oracle's representation (fp32, or bf16 bits as u16)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype == torch.float32:
        return f32(t)
    return t.detach().cpu().numpy()


def to_torch_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def fill_ranges(buf: torch.Tensor, db, values):
    """Write per-tensor values into their ranges of a flat buffer."""
    for t, v in enumerate(values):
        o = db.offsets[t]
        buf[o:o + v.numel()].copy_(v.reshape(-1))


def padding_mask(total: int, offsets, numel) -> np.ndarray:
    m = np.ones(total, bool)
    for o, n in zip(offsets, numel):
        m[o:o + n] = False
    return m


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    if got.dtype == np.float32:
        g, w = got.view(np.uint32), want.view(np.uint32)
        nan = np.isnan(got) & np.isnan(want)
        bad = (g != w) & ~nan
    else:
        bad = got != want
    if bad.any():
        idx = np.nonzero(bad)[0][:8]
        raise AssertionError(f"{what}: {int(bad.sum())} mismatches, first at {idx.tolist()}: "
                             f"got {got[idx].tolist()} want {want[idx].tolist()}")


def assert_norms_close(got_norms, got_total, want_norms, want_total, rel=1e-5, what="norm"):
    g = np.asarray(got_norms, np.float64)
    w = np.asarray(want_norms, np.float64)
    err = np.abs(g - w)
    ok = err <= rel * np.abs(w)
    if not ok.all():
        i = int(np.nonzero(~ok)[0][0])
        raise AssertionError(f"{what}: tensor {i} got {g[i]!r} want {w[i]!r} rel {err[i] / max(w[i], 1e-300):.3e}")
    assert abs(float(got_total) - want_total) <= rel * abs(want_total), (got_total, want_total)
