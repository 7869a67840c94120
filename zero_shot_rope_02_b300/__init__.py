"""Dynamic Bifocal RoPE attention for the NVIDIA B300 (sm_103a).

The compute lives in ``libjetlong.so`` (C ABI, ``include/jetlong.h``); this
package only marshals torch tensors into it (``binding``), builds it
(``build``) and draws seeded synthetic inputs (``inputs``).  The binding is
loaded on first use of any of its names, and that load fails loudly when the
library has not been built: there is no fallback path.
"""
_BINDING_NAMES = (
    "EXPORTS", "JetLongError", "LIB_PATH", "jl_bifocal_decode", "jl_bifocal_decode_workspace_size",
    "jl_bifocal_prefill", "jl_debug_grouped_positions", "jl_debug_status", "jl_debug_tile_classes",
    "jl_group_factor", "jl_rope_apply", "jl_version", "lib", "status_string",
    "jl_bifocal_decode_noalloc", "jl_debug_wait_timeout", "jl_bifocal_prefill_chunk",
    "jl_bifocal_decode_paged", "jl_bifocal_decode_paged_workspace_size", "jl_rope_cache_write",
    "jl_group_factor_ex", "jl_bifocal_prefill_ex", "jl_bifocal_decode_ex", "JL_VARIANT_PER_QUERY_G",
    "JL_VARIANT_SLIDING", "JL_VARIANT_QUERY_SHIFT", "JL_PREFILL_CTA_PAIR",
    "JL_PREFILL_ONE_CTA",
)

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
