"""Seeded synthetic workloads shared by the tests and the bench (no step arithmetic)."""
from .workloads import *  # noqa: F401,F403
