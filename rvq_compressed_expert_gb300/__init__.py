"""GB300-native routed-expert step of an RVQ-compressed Mixture-of-Experts layer.

The compute lives in libwaste_moe.so (CUDA, sm_103a) behind the C ABI of
include/waste_moe.h; ``binding`` is its ctypes binding, ``layer`` a helper that
holds one layer's weights on the GPU, ``synth`` the seeded synthetic inputs.
"""
from ._build import build  # noqa: F401

__all__ = ["build"]
