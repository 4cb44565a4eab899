"""GB300-native dynamic sparse attention: InfiniteHiP chunk-pruned decode and
MInference vertical-slash prefill, as hand-written sm_103a kernels behind a C ABI.

The Python surface mirrors the C entry points in ``include/dsa.h`` one to one;
it only marshals torch CUDA tensors into pointers.  Importing this package
does not load the library; the first call does, and raises if the library
has not been built (``__graft_entry__.build()``).
"""
from .binding import (  # noqa: F401
    DsaError,
    ashape_index_build,
    block_sparse_index_build,
    block_sparse_index_build_workspace_bytes,
    device_error,
    HipConfig,
    hip_max_chunks,
    hip_prefill_lists,
    hip_prefill_max_chunks,
    hip_prefill_select,
    hip_prefill_select_workspace_bytes,
    hip_select,
    hip_select_cached,
    HipSelectCache,
    hip_select_workspace_bytes,
    library_path,
    mixed_index_build,
    mixed_index_build_workspace_bytes,
    load,
    profile_collect,
    profile_enable,
    refresh_mask,
    set_wait_limit,
    sparse_attn_decode,
    sparse_attn_decode_noalloc,
    sparse_attn_decode_workspace_bytes,
    sparse_attn_prefill,
    vs_index_build,
    vs_index_build_workspace_bytes,
)
