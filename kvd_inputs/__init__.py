"""Seeded synthetic inputs for paged decode attention (random numbers and input structure only)."""

from . import gen, workloads
from .workloads import Workload, get, WORKLOADS

__all__ = ["gen", "workloads", "Workload", "get", "WORKLOADS"]
