"""CPU oracle for the NVFP4 block-scaled MoE path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may import
this package; the CUDA library never does.
"""
from . import nvfp4_oracle  # noqa: F401
