"""SAF (Selective Attention Freezing) hybrid causal attention for one GB300.

The compute path is ``libsaf.so`` (hand-written CUDA for sm_103a behind the C
ABI in ``include/saf.h``).  ``_binding`` marshals arguments to it through
ctypes; ``api`` wraps those calls for torch tensors (device memory and
streams only).  ``synthetic`` draws the seeded workloads.

Importing ``api`` or ``_binding`` fails loudly when the library is not built:
there is no CPU or PyTorch fallback.
"""

import importlib

__all__ = ["api", "synthetic", "build"]


def build(verbose: bool = False) -> str:
    from ._build import build as _b
    return _b(verbose=verbose)


def __getattr__(name):
    if name in ("api", "synthetic", "_binding"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
