"""GB300-native sliced tensor-parallel MLP (Domino-style communication overlap).

The compute runs in libdomino_gb300.so (hand-written CUDA for sm_103a behind
the C ABI of include/domino.h); ``binding`` marshals torch tensors into it and
loads the library on first use.  ``workloads`` holds the seeded synthetic inputs.
"""
from . import binding, workloads  # noqa: F401

__all__ = ["binding", "workloads"]
