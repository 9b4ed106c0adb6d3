"""GB300-native DBuffer group operators (sm_103a).

The data-parallel hot path of a RaggedShard/DBuffer FSDP on one GPU: a host C++
planner lays a tensor group out in one flat buffer of m shard slices without
cutting blocks, and hand-written CUDA kernels run each group operator (pack with
fused cast, unpack, gradient scale/accumulate/zero, ragged norm with non-finite
flag, block-wise FP8/INT8 quantisation) over the whole group, one launch per
operator (the norm adds a small finishing launch), never one per tensor.

``dbuf`` is the thin binding of the C ABI (include/dbuf.h); ``DBuffer`` wraps a
plan with PyTorch-managed device memory.
"""
from . import dbuf  # noqa: F401
from .dbuffer import DBuffer, dtype_code  # noqa: F401

__all__ = ["dbuf", "DBuffer", "dtype_code"]
