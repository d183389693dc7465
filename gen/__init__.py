"""Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests and the bench."""
from .inputs import (WORKLOADS, Workload, make_qkv, make_qkv_rising, sweep_points,  # noqa: F401
                     sweep_seed, to_dtype, workload)
