"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the oracle."""
from .synth import *  # noqa: F401,F403
