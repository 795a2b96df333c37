"""PagedAttention decode for GB300: a C-ABI CUDA library (libpagedattn.so)
and its thin Python binding.

    from paged_kv_cache_173_gb300 import api
    api.pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping)
    api.pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale)

``workloads`` builds seeded synthetic batches; it holds no attention
arithmetic.  The binding is imported lazily so that ``workloads`` can be used
without torch's CUDA runtime.
"""

__all__ = ["api", "workloads", "build"]
