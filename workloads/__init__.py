"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Holds no attention arithmetic: mask encoders (`masks`), the benchmark
workloads (`configs`) and seeded bf16 tensors (`tensors`).
"""
from . import configs, masks, tensors  # noqa: F401
