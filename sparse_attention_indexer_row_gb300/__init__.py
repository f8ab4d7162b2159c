"""Batched row-wise top-k selection for a sparse-attention indexer, on GB300.

The compute path is the CUDA library ``libtopk_gb300.so`` built from
``csrc/``; ``binding`` marshals arguments to its C ABI.  ``synth`` draws the
seeded workloads.  The binding is imported lazily so that the generators can
be used on a machine without the built library.
"""

import importlib

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name in ("binding", "synth", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
