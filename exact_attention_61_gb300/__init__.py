"""GB300 (sm_103a) fused exact scaled-dot-product attention forward.

The compute lives in ``libattn.so`` (hand-written sm_103a CUDA kernels behind the
C ABI of ``include/attn.h``); :mod:`.attn` is its ctypes binding. Importing this
package does not load the library; the first call does, and fails loudly if the
library has not been built.
"""
from . import counts  # noqa: F401  (host-side FLOP / traffic / schedule arithmetic)

__all__ = ["attn", "counts", "build"]


def __getattr__(name):
    if name in ("attn", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
