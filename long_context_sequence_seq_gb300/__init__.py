"""GB300-native single-GPU hot path of Ulysses sequence parallelism.

The all-to-all re-layouts and the local causal/varlen GQA attention run in
hand-written sm_103a CUDA kernels inside ``libulysses.so`` (C ABI declared in
``include/ulysses.h``); ``ulysses`` is the thin ctypes binding over it.
"""
from . import inputs  # noqa: F401  (seeded synthetic inputs; no method arithmetic)

__all__ = ["inputs", "ulysses", "build"]


def __getattr__(name):
    if name in ("ulysses", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
