"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds input generation only -- workload shapes, selection traces,
and KV record bytes.  It contains none of the cache's arithmetic (no LRU, no
page table, no victim choice), so the oracle and the CUDA path stay
independent while reading identical inputs.
"""
from .configs import WORKLOADS, Workload, get, sweep_workload, SWEEP_B, SWEEP_F  # noqa: F401
