"""Batched row-wise top-k selection for a sparse-attention indexer, on GB300.

The compute path is the CUDA library ``libtopk_gb300.so`` built from
``csrc/``; ``binding`` marshals arguments to its C ABI.  ``synth`` draws the
seeded workloads.  The binding is imported lazily so that the generators can
be used on a machine without the built library.
"""

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    raise AttributeError(name)
