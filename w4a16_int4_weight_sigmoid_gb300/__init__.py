"""GB300 (sm_103a) W4A16 INT4-weight MoE layer with sigmoid+bias routing.

The compute path is the CUDA library libchord_moe.so (C ABI in
include/chord_moe.h); `chord` is its thin ctypes binding and `layer` keeps
prepacked weights and workspace in torch-managed device memory.
"""
from . import workload  # noqa: F401

__all__ = ["workload", "chord", "layer", "build"]
