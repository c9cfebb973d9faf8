"""CPU float64 oracle for the paged-KV-cache hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package; the CUDA library never does.
"""
from .pkv_oracle import *  # noqa: F401,F403
