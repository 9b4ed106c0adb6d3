"""Independent checks of a DBuffer layout, written straight from the problem
statement of "veScale-FSDP: Flexible and High-Performance FSDP at Scale",
§5 Planning algorithm (problem formulation):

  minimise the per-shard size S over offsets l_t such that
   (i)   tensors keep the default order and do not overlap (padding only between
         tensors): l_t >= l_{t-1} + n_{t-1};
   (ii)  every offset is a multiple of the alignment a (and so is S);
   (iii) a shard boundary B_k strictly inside a tensor is a whole number of
         units g_t from the tensor's start (no block is split);
   (iv)  the last tensor ends inside the buffer: l_last + n_last <= B_m.

Shard k spans [U*c_k, U*c_{k+1}) with c_k the prefix sums of the per-shard units
(RaggedShard ``local_units``); even shards have all units 1 and U = S.

Nothing here is shared with the oracle or the CUDA path.  ``brute_force_plan``
assumes nothing about the structure of the optimum (no greedy argument): at each
candidate S it decides feasibility by dynamic programming over every aligned
start of every tensor.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np


def unit_of(rows: int, cols: int, gran_rows: int) -> int:
    n = rows * cols
    if gran_rows <= 0 or gran_rows >= rows:
        return n
    return gran_rows * cols


def boundaries(U: int, m: int, units: Optional[Sequence[int]]) -> List[int]:
    c = [0]
    for k in range(m):
        c.append(c[-1] + (units[k] if units is not None else 1))
    return [U * x for x in c]


def check_layout(specs, offsets, bounds, align) -> List[str]:
    """Return the list of violated constraints (empty = valid)."""
    errs = []
    m = len(bounds) - 1
    prev_end = 0
    for t, s in enumerate(specs):
        n = s.rows * s.cols
        g = unit_of(s.rows, s.cols, s.gran_rows)
        lt = int(offsets[t])
        if lt < prev_end:
            errs.append(f"(i) tensor {t} starts at {lt} before previous end {prev_end}")
        if lt % align:
            errs.append(f"(ii) tensor {t} offset {lt} not a multiple of {align}")
        for k in range(1, m):
            b = int(bounds[k])
            if lt < b < lt + n and (b - lt) % g:
                errs.append(f"(iii) boundary {k} at {b} splits a unit of tensor {t}")
        prev_end = lt + n
    if prev_end > int(bounds[-1]):
        errs.append(f"(iv) last tensor ends at {prev_end} past the buffer end {bounds[-1]}")
    for k in range(m + 1):
        if int(bounds[k]) % align:
            errs.append(f"(ii) boundary {k} not aligned")
    return errs


def _valid_starts(n: int, g: int, B: Sequence[int], align: int) -> np.ndarray:
    """Mask over p in [0, B_m] of starts satisfying (ii), (iii) and (iv) alone."""
    top = B[-1]
    p = np.arange(top + 1, dtype=np.int64)
    ok = (p % align == 0) & (p + n <= top)
    for b in B[1:-1]:
        inside = (p < b) & (b < p + n)
        ok &= ~(inside & ((b - p) % g != 0))
    return ok


def feasible_placement(specs, U, m, units, align) -> Optional[List[int]]:
    """Lexicographically smallest feasible offsets at unit size U, or None."""
    B = boundaries(U, m, units)
    top = B[-1]
    T = len(specs)
    ns = [s.rows * s.cols for s in specs]
    gs = [max(1, unit_of(s.rows, s.cols, s.gran_rows)) for s in specs]
    valid = [_valid_starts(ns[t], gs[t], B, align) for t in range(T)]
    # F[t][e]: tensors t.. can all be placed when the previous tensor ends at e.
    F = [None] * (T + 1)
    F[T] = np.ones(top + 1, dtype=bool)
    idx = np.arange(top + 1, dtype=np.int64)
    for t in range(T - 1, -1, -1):
        ends = idx + ns[t]
        good = valid[t].copy()
        inr = ends <= top
        good[inr] &= F[t + 1][ends[inr]]
        good[~inr] = False
        # any good start p >= e (alignment is already inside good)
        suffix = np.logical_or.accumulate(good[::-1])[::-1]
        F[t] = suffix
    if T and not F[0][0]:
        return None
    offs = []
    e = 0
    for t in range(T):
        ends = idx + ns[t]
        good = valid[t].copy()
        inr = ends <= top
        good[inr] &= F[t + 1][ends[inr]]
        good[~inr] = False
        cand = np.nonzero(good[e:])[0]
        p = e + int(cand[0])
        offs.append(p)
        e = p + ns[t]
    return offs


def brute_force_plan(specs, m, units=None, align=1, max_U=None) -> Tuple[int, List[int]]:
    """Smallest aligned U with a feasible placement, and its lexicographically
    smallest offsets.  Scans every multiple of `align` from 0."""
    E = sum(s.rows * s.cols for s in specs)
    hi = max_U if max_U is not None else E + len(specs) * align + align
    U = 0
    while U <= hi:
        offs = feasible_placement(specs, U, m, units, align)
        if offs is not None:
            return U, offs
        U += align
    raise AssertionError("no feasible U found below the trivial bound")


def naive_concat(specs, m, align=1):
    """The naive layout of Figure 6(a): tensors concatenated back to back, the
    buffer split into m equal shards with no regard for blocks."""
    offs, e = [], 0
    for s in specs:
        e = (e + align - 1) // align * align
        offs.append(e)
        e += s.rows * s.cols
    S = -(-e // m)
    S = (S + align - 1) // align * align
    return S, offs, [k * S for k in range(m + 1)]


def two_boundary_survivors(specs, sizes) -> np.ndarray:
    """The sizes S (even shards, boundaries at k*S) that this consequence of
    constraint (iii) leaves possible.  A tensor of n > 2S elements lies inside
    [0, m*S] and therefore holds two consecutive boundaries k*S and (k+1)*S
    strictly inside it; (iii) puts both a whole number of units g from its
    start, so g divides their distance S.  Any size failing that for some
    tensor has no layout at all.  A whole-tensor unit (g = n) never divides an
    S < n / 2, so such a tensor always rules the size out."""
    S = np.asarray(sizes, dtype=np.int64)
    ok = np.ones(len(S), dtype=bool)
    for s in specs:
        n = s.rows * s.cols
        if n == 0:
            continue
        g = max(1, min(unit_of(s.rows, s.cols, s.gran_rows), n))
        ok &= ~((n > 2 * S) & (S % g != 0))
    return S[ok]


def literal_greedy(specs, U, m, units, align, window=512) -> Optional[List[int]]:
    """Greedy-leftmost offsets at unit size U by a literal scan, or None.

    Each tensor starts at the smallest aligned p >= the previous tensor's end
    such that the tensor ends inside the buffer (iv) and every boundary strictly
    inside [p, p + n) lies a multiple of g_t from p (iii).  The candidate starts
    are examined in increasing order, a window of them at a time (vectorised);
    nothing is skipped by reasoning about the constraint's structure.
    """
    B = np.asarray(boundaries(U, m, units), dtype=np.int64)
    top = int(B[-1])
    inner = B[1:-1]
    offs: List[int] = []
    e = 0
    for s in specs:
        n = s.rows * s.cols
        g = max(1, unit_of(s.rows, s.cols, s.gran_rows))
        p0 = -(-e // align) * align
        found = None
        w = window
        while p0 + n <= top:
            cand = p0 + align * np.arange(w, dtype=np.int64)
            cand = cand[cand + n <= top]
            if cand.size == 0:
                break
            ok = np.ones(cand.size, dtype=bool)
            near = inner[(inner > cand[0]) & (inner < cand[-1] + n)]
            for b in near:
                ok &= ~((cand < b) & (b < cand + n) & ((b - cand) % g != 0))
            hit = np.flatnonzero(ok)
            if hit.size:
                found = int(cand[hit[0]])
                break
            p0 = int(cand[-1]) + align
            w = min(2 * w, 1 << 21)
        if found is None:
            return None
        offs.append(found)
        e = found + n
    return offs
