"""Seeded synthetic workloads shared by the oracle tests, the CUDA tests and the bench.

Holds shapes and random-input recipes only; no arithmetic of the verify step.
"""
from .configs import (BLOCK, ROWS, ModelShape, Workload, WORKLOADS, WORKLOAD_ORDER,
                      TINY, HALF_B_BF16, HALF_B_MIXED, SEVEN_B_MIXED, linear_shapes,
                      DRAFTER_LAYERS, drafter_shape, mask_token)
from . import gen
