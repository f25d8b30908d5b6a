"""Per-rank context-parallel blockwise attention for GB300 (sm_103a).

Python binding of ``libcpattn.so`` (C ABI in ``include/cpattn.h``).  The binding only checks and
marshals arguments; every step of the computation runs in the library's CUDA kernels.  PyTorch
is used for device memory and streams.  The shared library is loaded on first use and a missing
or unloadable library raises -- there is no CPU fallback.
"""

from .api import (  # noqa: F401
    CpError,
    PosMap,
    shard_layout,
    shard_segments,
    sub_chunk_map,
    partial_attn,
    partial_attn_chunks,
    merge_partials,
    attn_bwd_prep,
    partial_attn_bwd,
    partial_attn_bwd_chunks,
    partial_attn_bwd_noalloc,
    NOALLOC_AUX_MAX_FLOATS,
    bwd_aux_floats,
    ulysses_reshard,
    library_path,
    load_library,
    version,
)

__all__ = [
    "CpError",
    "PosMap",
    "shard_layout",
    "shard_segments",
    "sub_chunk_map",
    "partial_attn",
    "partial_attn_chunks",
    "merge_partials",
    "attn_bwd_prep",
    "partial_attn_bwd",
    "partial_attn_bwd_chunks",
    "partial_attn_bwd_noalloc",
    "NOALLOC_AUX_MAX_FLOATS",
    "bwd_aux_floats",
    "ulysses_reshard",
    "library_path",
    "load_library",
    "version",
]
