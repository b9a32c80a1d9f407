"""GB300 (sm_103a) attention forward pass: a tiled online softmax with TMA loads, tcgen05 MMAs
and tensor-memory accumulators, behind the C interface of include/fa.h.

``fa``      -- the ctypes binding (``forward``, ``forward_host``, raw ``fa_fwd``).
``build``   -- compiles ``csrc/`` into ``libfa.so`` with nvcc.
``inputs``  -- seeded synthetic workloads (no attention arithmetic).
"""
from . import inputs  # noqa: F401  (no GPU or library needed)


def __getattr__(name):
    if name in ("fa", "build"):
        import importlib

        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
