"""GB300-native hot path of precomputed-KV RAG: span gather + RoPE
re-rotation + stitch, and query prefill attention over the stitched prefix.

The compute runs in libkvr.so (hand-written sm_103a CUDA behind the C ABI in
include/kvr.h); :mod:`.kvr` is its ctypes binding, :mod:`.workloads` the
seeded synthetic inputs, :mod:`.build` the in-tree nvcc build.
"""
from . import workloads  # noqa: F401

__all__ = ["kvr", "workloads", "build"]
