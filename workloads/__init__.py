"""Seeded synthetic inputs for the paged-KV attention step.

This package is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds random draws and the block bookkeeping that defines
the inputs (physical block ids, block tables, slot numbers, sequence
boundaries), and none of the method's arithmetic: no normalisation, no RoPE,
no attention.
"""

from .synthetic import (  # noqa: F401
    BLOCK_SIZE,
    HEAD_DIM,
    NAN_BF16,
    NUM_KV_HEADS,
    NUM_Q_HEADS,
    Workload,
    build_workload,
    config_workload,
    CONFIG_NAMES,
    bf16_bits_from_f32,
)
