"""GB300-native MoE token dispatch / combine data movement.

The compute path is the CUDA library ``libep_gb300.so`` built from ``csrc/``
for sm_103a; ``combine_movement_gb300.ep`` is its thin Python binding (same
names as the C ABI in ``include/ep.h``). Importing the binding loads the
library and raises if it is missing: there is no CPU fallback.
"""
import importlib

__all__ = ["ep", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
