"""GB300-native paged KV-cache decode path.

CUDA kernels for sm_103a behind a C ABI (``include/paged_attention.h``):
slot mapping, reshape_and_cache, paged decode attention with an optional
split-context partition pass and merge, and copy-on-write block copies.
This package is the thin Python binding over that library plus the seeded
workload generator used by the tests and the benchmark.

The binding is imported lazily so that the workload generator can be used on
machines without the built library; any call into the binding raises if the
CUDA library is missing -- there is no CPU fallback.
"""
from __future__ import annotations

__all__ = [
    "pa_slot_mapping", "pa_reshape_and_cache", "pa_copy_blocks",
    "pa_decode_attention", "pa_decode_workspace_bytes", "PAError",
    "pa_reshape_and_cache_fp8", "pa_decode_attention_fp8", "pa_decode_attention_noalloc",
    "library_path",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
