"""load_balancing_gb300 -- load-balanced block-sparse attention forward on one GB300.

The product is the C-ABI shared library ``libdbsp.so`` (declared in
``include/dbsp.h``, built from ``csrc/`` for sm_103a). ``dbsp`` is its thin Python
binding: it marshals torch tensors into pointers and streams and does nothing
else. Every step of the path runs in the library's CUDA kernels; there is no CPU
fallback, and calling the binding without the built library raises.

``workloads`` generates the seeded synthetic inputs (masks, Q/K/V, KV shards).
"""

from . import workloads  # noqa: F401

__all__ = ["workloads", "dbsp"]


def __getattr__(name):
    if name in ("dbsp", "path", "build"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
