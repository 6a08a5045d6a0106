"""Packed multi-adapter LoRA layer (forward, backward, AdamW) for GB300 (sm_103a).

The compute lives in ``libmlora.so`` (C ABI in ``include/mlora.h``); ``_mlora`` is its ctypes
binding and ``layer.PackedLoRA`` holds the device buffers of one pack.  ``workloads`` draws the
seeded synthetic inputs.  Importing the package does not load the CUDA library; the first call
that needs it does, and fails loudly if it has not been built.
"""
from . import _mlora  # noqa: F401

__all__ = ["_mlora", "layer", "workloads", "build"]
