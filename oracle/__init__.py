"""CPU oracle of the Stable LatentMoE forward with Quantile Balancing.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py, never by the product path.
"""
from .qb_oracle import *  # noqa: F401,F403
