"""The data-parallel exchange around the DBuffer group operators on m ranks.

"veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer and
Figure 7: parameters are all-gathered and gradients reduce-scattered in place on
the planned flat buffer, each rank owning one shard slice of it, so no copy sits
between a tensor and the collective; §4 and §6.3: no block crosses a shard, so
each rank's block quantisation needs only its slice.  "PyTorch FSDP:
Experiences on Scaling Fully Sharded Data Parallel", FlatParameter: the
collectives want equal shard sizes, which an even plan gives (S per rank);
native mixed precision: the fp32 master shard is cast to bf16 before the
AllGather; sharded gradient scaler: the non-finite flag is reduced across ranks.

Rank k of m (world size m, even shards, slice k = [k*S, (k+1)*S)):

  gradients   copy-in of the rank's gradient tensors into its m*S buffer
              -> ReduceScatter (sum) into its S slice
              -> scale/accumulate/zero on the slice (scale 1/m makes the sum a mean)
              -> per-tensor sums of squares and non-finite flag of the accumulator slice
              -> AllReduce (sum) of the sums, AllReduce (max) of the flag -> norms
              -> block quantisation of the accumulator slice (local codes and scales)
  parameters  cast of the rank's piece of every fp32 master tensor into its bf16 slice
              -> AllGather of the slices into the m*S bf16 buffer
              -> copy-out into the bf16 compute tensors

Every step of the arithmetic runs in the group operators of `full` (the plan of
the whole buffer) and `local` (the plan of this rank's slice, DBuffer.slice(k));
this module only orders them around the torch.distributed collectives.  Any
pair of objects with DBuffer's operator methods can be passed in.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch
import torch.distributed as dist


class ShardedStep:
    """The exchange of one planned tensor group on `world` ranks."""

    def __init__(self, full, local, rank: int, world: int, group=None):
        if full.m != world:
            raise ValueError(f"the plan has {full.m} shards for {world} ranks")
        sizes = {full.shard_bounds[k + 1] - full.shard_bounds[k] for k in range(full.m)}
        if len(sizes) != 1:
            raise ValueError("the exchange needs equal shard sizes (an even plan)")
        if local.total != full.S:
            raise ValueError("the local plan is not one shard of the full plan")
        self.full = full
        self.local = local
        self.rank = rank
        self.world = world
        self.group = group

    # -- gradients ---------------------------------------------------------------
    def reduce_gradients(self, grads: Sequence[torch.Tensor], grad_full: torch.Tensor,
                         grad_local: torch.Tensor, acc_local: torch.Tensor, scale: float,
                         codes: Optional[torch.Tensor] = None,
                         scales: Optional[torch.Tensor] = None):
        """Copy-in, ReduceScatter, accumulate, sharded norm and block quantisation.

        grad_full: the rank's m*S gradient buffer (padding zero); grad_local and
        acc_local: its S slice buffers (same dtype as grad_full; fp32).  Returns
        (tensor_norms, total_norm, nonfinite, codes, scales); codes and scales are
        None when the slice holds no quantised block."""
        self.full.pack_cast(grads, grad_full)
        dist.reduce_scatter_tensor(grad_local, grad_full, op=dist.ReduceOp.SUM, group=self.group)
        self.local.scale_accum_zero(grad_local, acc_local, scale)
        sumsq, flag = self.local.norm_sumsq(acc_local)
        dist.all_reduce(sumsq, op=dist.ReduceOp.SUM, group=self.group)
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=self.group)
        norms, total = self.local.norm_finish(sumsq)
        if self.local.n_scales:
            codes, scales = self.local.block_quant(acc_local, codes=codes, scales=scales)
        else:
            codes = scales = None
        return norms, total, flag, codes, scales

    # -- parameters ---------------------------------------------------------------
    def gather_parameters(self, master: Sequence[torch.Tensor], buf_local: torch.Tensor,
                          buf_full: torch.Tensor, compute: Sequence[torch.Tensor]) -> None:
        """Cast the rank's piece of each master tensor into its slice, AllGather the
        slices, copy out every compute tensor.  The AllGather moves the slices'
        bytes unchanged (as bytes, whatever the buffer's element type)."""
        self.local.pack_cast(master, buf_local)
        dist.all_gather_into_tensor(buf_full.view(torch.uint8), buf_local.view(torch.uint8),
                                    group=self.group)
        self.full.unpack(buf_full, compute)
