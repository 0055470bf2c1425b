"""Test infrastructure: the fp64 CPU oracle of the MoE layer (see moe_oracle.py).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this package.
"""
from .moe_oracle import *  # noqa: F401,F403
