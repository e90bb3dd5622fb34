"""GB300-native chunked gated-delta-rule prefill forward.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI
declared in ``include/gdn.h`` (``libgdn.so``). This package is a thin
binding over that library: it marshals torch tensors to device pointers and
calls the ABI; every step of the method runs in the kernels. Importing the
package loads nothing; the first call loads ``libgdn.so`` and raises if it is
missing (there is no CPU fallback).
"""
from __future__ import annotations

__all__ = [
    "gdn_chunk_fwd", "gdn_build_chunk_indices", "gdn_workspace_size",
    "gdn_read_status", "gdn_status_string", "GdnError", "load_library",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
