"""Seeded synthetic inputs (shapes and value distributions only, no decoder math)."""
from .workloads import (  # noqa: F401
    WORKLOADS, Workload, generate, custom, to_host, kv_buffer, BF16, AFFINE4_G64, AFFINE8_G64, GROUP,
)
