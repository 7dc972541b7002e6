"""Seeded synthetic inputs for the MoE layer (shared by tests and bench).

This module only draws random inputs; it holds none of the layer's
arithmetic.  Both the CUDA path and the float64 oracle receive exactly the
arrays made here.
"""
from .workloads import (WORKLOADS, SWEEP_TOKENS, SWEEP_ROUTINGS, Workload,  # noqa: F401
                        sweep_workload, make_logit_offset, make_router_weight,
                        make_x, make_weights, seeds_for)
