"""Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests and the bench."""
from .inputs import (WORKLOADS, Workload, make_qkv, sweep_points, sweep_seed,  # noqa: F401
                     to_dtype, workload)
