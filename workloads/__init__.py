"""Seeded synthetic inputs shared by tests, bench and smoke (no method arithmetic)."""
from .gen import *  # noqa: F401,F403
from .gen import PosCfg, Workload, make_workload, make_custom, WORKLOADS, f32_to_bf16_bits  # noqa: F401
