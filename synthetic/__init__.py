"""Seeded synthetic inputs (shapes and value distributions only, no decoder math)."""
from .workloads import WORKLOADS, Workload, generate, custom, to_host, BF16, AFFINE4_G64, GROUP  # noqa: F401
