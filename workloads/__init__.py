"""Seeded synthetic workloads shared by the CUDA path's tests/benchmark and the CPU oracle's tests."""
from .synth import WORKLOADS, BY_NAME, Workload  # noqa: F401
