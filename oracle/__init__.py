"""CPU float64 oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and the
oracle never imports the CUDA library.  Every function here is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle.py`` (brute force, closed forms,
invariants and library routines); none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    attention_weights,
    gather_tokens,
    merge_states,
    mla_decode,
    paged_decode,
    paged_decode_split,
    paged_prefill,
    paged_prefill_rows,
    softmax_attention,
    split_partials,
)
from .cache_write import mla_reshape_and_cache, reshape_and_cache  # noqa: F401,E402
from .prefix_cache import block_hashes, lookup_or_allocate, mix64  # noqa: F401,E402
