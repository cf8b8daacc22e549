"""GB300-native routed-expert step of an RVQ-compressed Mixture-of-Experts layer.

The compute lives in libwaste_moe.so (CUDA, sm_103a) behind the C ABI of
include/waste_moe.h.  Modules:

- ``binding``: the ctypes binding of that C ABI (argument marshalling only);
- ``layer``:   ``MoELayer``, one layer's router, codebooks and packed records on the GPU;
- ``stack``:   ``DecodeStack``, a stack of layers decoded with the next-layer lookahead;
- ``bank``:    ``TieredStack``, layers whose records live in pinned host memory behind an
  HBM cache (the tiered expert bank, with read/compute overlap);
- ``trace``:   ``RouteTrace``, the routing of a stack run as JSON lines;
- ``synth``:   seeded synthetic inputs of the workloads' shapes.

``build()`` compiles the library in-tree; every call fails loudly when it is missing.
"""
from ._build import build  # noqa: F401

__all__ = ["build"]
