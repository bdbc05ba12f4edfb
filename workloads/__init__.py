"""Seeded synthetic inputs for paged-KV decode attention.

This package only draws random numbers and lays them out in the paged pool
format; it contains none of the attention arithmetic. Both the CPU oracle
(tests) and the CUDA library (tests, bench) consume what it produces.
"""
from .configs import CONFIGS, WorkloadSpec, spec_by_name  # noqa: F401
from .gen import Workload, make_workload, make_append_batch, KV_BF16, KV_FP8, KV_MLA656, KV_F64  # noqa: F401
