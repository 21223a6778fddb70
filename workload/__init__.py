"""Seeded synthetic inputs for the MoE verify step (shared by tests, bench and oracle checks)."""
from .gen import CONFIGS, MoEConfig, Workload, make_workload, small_case  # noqa: F401
