"""Seeded synthetic workloads (shapes and input generators) for the DFlash draft-and-verify step.

Used by both the oracle side (tests, CPU baseline) and the CUDA side (tests, bench).
It holds none of the method's arithmetic.
"""
from .configs import (DrafterShape, Workload, TINY, QWEN3_8B, LLAMA31_8B, W_TINY, W_QWEN3_8B,
                      W_SWEEP, W_BATCHED, W_LLAMA, WORKLOADS, weight_bytes)
