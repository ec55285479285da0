"""GB300 (sm_103a) NVFP4 block-scaled MoE expert path: C-ABI library + thin torch binding.

The compute path is the shared library built from ``csrc/`` (see ``build.py``);
``ops`` marshals torch tensors into its entry points and ``workloads`` makes
the seeded synthetic inputs.
"""

__all__ = ["ops", "workloads", "build"]
