"""Paged KV-cache decode attention for NVIDIA GB300 (sm_103a).

The compute lives in the C-ABI library ``libpa_gb300.so`` (``include/pa.h``); this package
holds its build script (:mod:`.build`), the ctypes binding (:mod:`.native`) and the seeded
synthetic workloads used by the tests and the benchmark (:mod:`.workloads`).

``from paged_kv_cache_table_gb300 import pa_decode_attention`` loads the library on first
use and raises if it has not been built; nothing falls back to another implementation.
"""

__version__ = "0.1.0"

_BINDING_NAMES = {
    "pa_kv_append", "pa_kv_append_tokens", "pa_block_copy", "pa_decode_workspace_size",
    "pa_decode_attention", "pa_decode_attention_noalloc", "pa_prefill_attention",
    "pa_status_string", "make_desc", "BlockManager", "PaError", "CacheDesc",
    "lib", "status_string", "PrefixCache", "block_hashes",
}


def __getattr__(name):
    if name in _BINDING_NAMES or name.startswith(("PA_", "pa_")):
        from . import native
        return getattr(native, name)
    raise AttributeError(name)
