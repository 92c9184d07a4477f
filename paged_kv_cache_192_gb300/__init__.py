"""GB300-native (sm_103a) PagedAttention: paged KV cache ops behind a C ABI.

* ``ops``            reshape_and_cache, copy_blocks, decode (split-KV),
                     prefill_chunk -- thin torch binding of include/pa.h
* ``block_manager``  native host block manager (free list, refcounts, CoW)
* ``layout``         slot arithmetic, pool allocation and filling
* ``synth``          seeded synthetic workloads (inputs only)
* ``build``          compiles csrc/ into libpa_gb300.so for sm_103a
"""
from . import synth  # noqa: F401  (no CUDA needed)

__all__ = ["ops", "block_manager", "layout", "synth", "build"]


def __getattr__(name):
    if name in ("ops", "block_manager", "layout", "build", "_lib"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
