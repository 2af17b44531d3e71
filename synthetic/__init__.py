"""Seeded synthetic workloads shared by the oracle and the CUDA path."""
from .workloads import *  # noqa: F401,F403
