"""Seeded synthetic workloads shared by the GPU path's tests/bench and the oracle.

Holds input generation only; none of the method's arithmetic lives here.
"""
from . import gen, configs  # noqa: F401
