"""CPU oracle for the prefix-cache block lookup -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; it shares no code with the CUDA library.

What it computes.  Prefix caching lets a new prompt reuse the KV pages of an
earlier prompt with the same leading tokens (vllm-metis 0.1.0 page,
"How the model maps onto vLLM", "Caches": vLLM's cache manager runs prefix
caching; "Status": 576 to 640 of 700 prompt tokens served from the cache).  A
page is found by a key that identifies the page's tokens *and everything
before them*:

1. Block hash.  For sequence s with tokens t_0 .. t_{L-1} and page size bs,
   full page b (tokens b*bs .. b*bs + bs - 1) gets
       local_b = fold of its tokens:  x = SEED;  x = mix64(x XOR t)  per token
       key_b   = mix64(key_{b-1} XOR local_b),  key_{-1} = 0  (0 is remapped to 1)
   where mix64 is the splitmix64 output function (Steele, Lea and Flood, "Fast
   splittable pseudorandom number generators", 2014) and SEED its golden-ratio
   increment 0x9E3779B97F4A7C15.  The partial last page has no key.
2. Lookup or allocate, in page order over the batch (sequence-major): a key
   already in the table is a hit (its page is reused, its reference count goes
   up by one); a new key takes the page on top of the free stack (reference
   count 1) and enters the table.  A key repeated inside the batch is new only
   at its first occurrence.  With the free stack empty a new key gets page -1
   and does not enter the table.
"""

from __future__ import annotations

import numpy as np

MASK = (1 << 64) - 1
SEED = 0x9E3779B97F4A7C15


def mix64(z: int) -> int:
    """splitmix64's output function (the generator's state increment is SEED)."""
    z &= MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def block_hashes(token_ids, cu_tokens, block_size: int) -> list:
    """Chained keys of every full page of every sequence, sequence-major (step 1)."""
    toks = np.asarray(token_ids, dtype=np.int64)
    cu = np.asarray(cu_tokens, dtype=np.int64)
    keys = []
    for s in range(len(cu) - 1):
        seq = toks[cu[s]:cu[s + 1]]
        key = 0
        for b in range(len(seq) // block_size):
            local = SEED
            for t in seq[b * block_size:(b + 1) * block_size]:
                local = mix64(local ^ (int(t) & 0xFFFFFFFF))
            key = mix64(key ^ local)
            if key == 0:
                key = 1
            keys.append(key)
    return keys


def lookup_or_allocate(keys, table: dict, free_stack: list, refcount: np.ndarray):
    """Step 2, one key at a time in order.  Returns ``(pages, hits, table, free_stack,
    refcount)``; the inputs are not modified."""
    table = dict(table)
    free_stack = list(free_stack)
    refcount = np.array(refcount, dtype=np.int64, copy=True)
    pages, hits = [], []
    for k in keys:
        if k in table:
            p = table[k]
            refcount[p] += 1
            pages.append(p)
            hits.append(True)
        elif free_stack:
            p = free_stack.pop()
            table[k] = p
            refcount[p] = 1
            pages.append(p)
            hits.append(False)
        else:
            pages.append(-1)
            hits.append(False)
    return pages, hits, table, free_stack, refcount
