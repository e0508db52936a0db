"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This package draws keys, values and queries and rounds them to their storage
dtype.  It holds none of the metered-decode arithmetic (no quantizer, witness,
meter or gate); both sides of every parity test receive exactly these arrays.
"""
from .gen import (  # noqa: F401
    HEAD_DIM,
    WORKLOADS,
    Workload,
    bf16_bits,
    bf16_from_bits,
    bf16_round,
    gen_append_kv,
    gen_kv,
    gen_q,
    planted_positions,
    sweep_workload,
)
