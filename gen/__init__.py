"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle."""
from .msa_inputs import *  # noqa: F401,F403
