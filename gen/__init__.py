"""Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests and the bench."""
from .inputs import (DECODE_WORKLOADS, WORKLOADS, DecodeWorkload, Workload,  # noqa: F401
                     decode_workload, make_qkv, make_qkv_kv, make_qkv_rising, sweep_points,
                     sweep_seed, to_dtype, workload)
