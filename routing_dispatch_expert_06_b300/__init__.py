"""B300-native forward pass of one Mixture-of-Experts layer.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI
declared in ``include/moe.h`` (``libmoe.so``).  The Python layer in
``routing_dispatch_expert_06_b300.moe`` only marshals arguments (torch
tensors for device memory and streams) into that library; importing this
package does not load it until a binding is used.
"""

import importlib

__all__ = ["inputs", "moe", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
