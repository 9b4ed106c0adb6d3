"""Seeded synthetic workloads for the DBuffer group operators.

This package only describes tensor groups (shapes, shard granularity, quantisation
blocks) and draws seeded random values for them.  It holds none of the layout or
group-operator arithmetic: the planner, the kernels and the oracle each do that on
their own.  Both the CUDA path's tests/bench and the oracle's tests take their
inputs from here.
"""
from .configs import (  # noqa: F401
    TensorSpec,
    GroupSpec,
    Workload,
    WORKLOADS,
    workload,
    param_values,
    grad_values,
    inf_injection,
)
