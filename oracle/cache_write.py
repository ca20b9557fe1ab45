"""CPU oracle for the KV-cache write -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; it shares no code with the CUDA library.

What it computes.  In front of every attention call the step's new keys and
values are written into the pages that the attention kernels then read
through the block table: vLLM's cache manager owns one paged KV cache layer
per attention layer (vllm-metis 0.1.0 page, "How the model maps onto vLLM",
"Caches"), and the scheduler's block table addresses those pages (vllm-metal
article, section 4).  A destination is a slot ``block_id * block_size +
offset``; a negative slot marks a padding token that is not written.  The
write is a copy, so the oracle is that copy written out token by token:

    k_cache[slot // block_size, slot % block_size] = key[n]
    v_cache[slot // block_size, slot % block_size] = value[n]

and for MLA (vllm-metal article, section 3: one latent cache, rows
``[c_kv | k_pe]``):

    kv_cache[slot // block_size, slot % block_size] = concat(kv_c[n], k_pe[n])

Tensors are CPU torch tensors (NumPy has no bf16); the caches are returned
as modified copies, the inputs are left untouched.
"""

from __future__ import annotations

import torch


def _slots(slot_mapping) -> list:
    if isinstance(slot_mapping, torch.Tensor):
        return [int(x) for x in slot_mapping.detach().cpu().tolist()]
    return [int(x) for x in slot_mapping]


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping):
    """Copies of ``k_cache`` / ``v_cache`` ([nb, bs, G, D]) with token ``n``'s
    rows ``key[n]`` / ``value[n]`` ([G, D]) written at ``slot_mapping[n]``.

    Slots below zero are skipped; a slot past the pool raises IndexError.
    """
    kc = k_cache.detach().cpu().clone()
    vc = v_cache.detach().cpu().clone()
    bs = kc.shape[1]
    total = kc.shape[0] * bs
    key = key.detach().cpu()
    value = value.detach().cpu()
    for n, slot in enumerate(_slots(slot_mapping)):
        if slot < 0:
            continue
        if slot >= total:
            raise IndexError("slot outside the block pool")
        kc[slot // bs, slot % bs] = key[n]
        vc[slot // bs, slot % bs] = value[n]
    return kc, vc


def mla_reshape_and_cache(kv_c: torch.Tensor, k_pe: torch.Tensor, kv_cache: torch.Tensor, slot_mapping):
    """Copy of ``kv_cache`` ([nb, bs, d_latent + d_rope]) with row
    ``concat(kv_c[n], k_pe[n])`` written at ``slot_mapping[n]`` (negative: skipped)."""
    kc = kv_cache.detach().cpu().clone()
    bs = kc.shape[1]
    total = kc.shape[0] * bs
    d_latent = kv_c.shape[-1]
    kv_c = kv_c.detach().cpu()
    k_pe = k_pe.detach().cpu()
    for n, slot in enumerate(_slots(slot_mapping)):
        if slot < 0:
            continue
        if slot >= total:
            raise IndexError("slot outside the block pool")
        kc[slot // bs, slot % bs, :d_latent] = kv_c[n]
        kc[slot // bs, slot % bs, d_latent:] = k_pe[n]
    return kc
