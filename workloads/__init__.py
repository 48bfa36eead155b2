"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Holds no attention arithmetic: mask encoders (`masks`), the benchmark
workloads (`configs`), seeded bf16 tensors (`tensors`) and chunk-load
instances for the chunk balancer (`chunks`).
"""
from . import chunks, configs, masks, tensors  # noqa: F401
