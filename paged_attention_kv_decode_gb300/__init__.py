"""GB300-native attention over a paged KV cache.

The compute lives in ``lib/libmetis_attn.so`` (hand-written CUDA for sm_103a,
C ABI declared in ``include/metis_attn.h``); this package holds its ctypes
binding, the in-tree build script and the seeded workload generator.  The
library is loaded on first use; a missing library raises instead of falling
back to any other implementation.
"""

from ._binding import (  # noqa: F401
    LIB_PATH,
    METIS_BF16,
    METIS_F32,
    SIGNATURES,
    STATUS_BAD_BLOCK_ID,
    STATUS_BAD_OFFSETS,
    STATUS_BAD_Q_LEN,
    STATUS_OUT_OF_PAGES,
    STATUS_SEQ_TOO_LONG,
    STATUS_TABLE_FULL,
    STATUS_WAIT_TIMEOUT,
    MetisError,
    load_library,
    metis_decode_workspace_bytes,
    metis_last_error,
    metis_merge_attn_states,
    metis_mla_decode,
    metis_mla_reshape_and_cache,
    metis_mla_workspace_bytes,
    NOALLOC_SCRATCH_BYTES,
    metis_paged_attn_decode,
    metis_paged_attn_decode_noalloc,
    metis_paged_attn_decode_partials,
    metis_paged_attn_prefill_chunk,
    metis_prefill_workspace_bytes,
    metis_prefix_block_hashes,
    metis_prefix_lookup,
    metis_prefix_lookup_workspace_bytes,
    metis_prefix_table_init,
    prefix_table_alloc,
    split_workspace_views,
    metis_read_status,
    metis_debug_wait_probe,
    metis_reshape_and_cache,
    metis_version,
)
from .pipeline import DecodePipeline  # noqa: F401,E402
