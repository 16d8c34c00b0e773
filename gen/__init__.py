"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the bench.

Holds input generation only: workload shapes (`configs`), draft-tree shapes
(`trees`), full input sets (`inputs`) and Monte-Carlo trial batches (`mc`).
"""
from .configs import Workload, WORKLOADS, get  # noqa: F401
