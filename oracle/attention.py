"""CPU float64 oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it.  It shares no code with the CUDA library.

What it computes.  The plugin pages (vllm-metal article, sections 3 and 4;
vllm-metis "How the model maps onto vLLM", "Caches") name the operation --
paged attention and MLA kernels fed by vLLM's block tables and sequence
lengths, prefix caching and chunked prefill -- without writing its formula.
The oracle therefore takes the plainest reading, textbook scaled-dot-product
softmax attention of each query row over the keys its sequence has cached,
and writes that definition out directly:

1. Walk the block table: logical token ``t`` of sequence ``s`` sits in
   physical block ``block_table[s, t // block_size]`` at slot
   ``t % block_size`` (vllm-metal article, section 4: the scheduler's block
   table and sequence lengths drive the kernel).
2. q head ``h`` reads kv head ``h // (H / G)`` (grouped-query attention with
   contiguous groups; the vllm-metis "Status" section runs GQA 4:1).
3. A query row at position ``p`` sees keys ``t <= p``; a chunk of ``q_len``
   new tokens of a sequence of ``L`` cached tokens holds positions
   ``L - q_len .. L - 1`` (vllm-metis "Status": chunked prefill and
   prefix-cache hits give the same result as an unchunked pass).
4. ``z_t = scale * q . k_t``; ``w = exp(z - max z) / sum exp(z - max z)``;
   ``out = sum_t w_t v_t``; ``lse = max z + ln sum exp(z - max z)``.
5. MLA (vllm-metal article, section 3): one latent head shared by all q
   heads; the key is the full ``d_latent + d_rope`` row, the value its first
   ``d_latent`` columns.
6. Split-KV: the same softmax over each partition of a sequence's tokens,
   then the log-sum-exp merge of the partial results.

Inputs are NumPy arrays or CPU torch tensors (NumPy has no bf16); the rows
that are used are converted to float64 exactly (bf16 and fp32 values are
representable).
No blocking, fusion or reordering beyond a library matrix product per
(sequence, kv head).
"""

from __future__ import annotations

import numpy as np
import torch

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """float64 copy of an array or a torch tensor (bf16 and fp32 values convert exactly)."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _arr(x):
    """Index-only access: torch tensors stay tensors (NumPy has no bf16), the rest become arrays."""
    return x if isinstance(x, torch.Tensor) else np.asarray(x)


def _ints(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().numpy()
    return np.asarray(x)


def gather_tokens(cache: np.ndarray, block_table_row: np.ndarray, seq_len: int, block_size: int) -> np.ndarray:
    """Rows ``cache[block_table_row[t // bs], t % bs]`` for ``t = 0 .. seq_len - 1``.

    Step 1 above.  ``cache`` is ``[num_blocks, block_size, ...]``; the result
    keeps the trailing dimensions.  Only the first ``ceil(seq_len / bs)``
    table entries are read, and only slots below ``seq_len``.
    """
    t = np.arange(int(seq_len))
    phys = _ints(block_table_row)[t // block_size].astype(np.int64)
    slot = t % block_size
    if len(t) and (phys.min() < 0 or phys.max() >= cache.shape[0]):
        raise IndexError("block table entry outside the block pool")
    if isinstance(cache, torch.Tensor):
        return cache[torch.from_numpy(phys), torch.from_numpy(slot)]
    return cache[phys, slot]


def softmax_attention(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float,
                      visible: np.ndarray):
    """Textbook softmax attention of each query row over its visible keys.

    ``q_rows`` [n, Dk], ``keys`` [L, Dk], ``values`` [L, Dv]; row ``i`` sees
    keys ``0 .. visible[i] - 1``.  Returns ``(out [n, Dv], lse [n])`` with
    the natural-log log-sum-exp of the scaled scores; a row with no visible
    key gives ``out = 0`` and ``lse = -inf``.
    """
    q_rows, keys, values = _f64(q_rows), _f64(keys), _f64(values)
    n = q_rows.shape[0]
    L = keys.shape[0]
    out = np.zeros((n, values.shape[1]), dtype=np.float64)
    lse = np.full(n, NEG_INF, dtype=np.float64)
    if L == 0 or n == 0:
        return out, lse
    visible = np.minimum(np.asarray(visible, dtype=np.int64), L)
    rows = visible > 0
    if not rows.any():
        return out, lse
    seen = np.arange(L)[None, :] < visible[rows, None]       # [n', L]
    z = float(scale) * (q_rows[rows] @ keys.T)                # [n', L]
    z = np.where(seen, z, NEG_INF)                            # hidden keys weigh exp(-inf) = 0
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    l = e.sum(axis=1)
    out[rows] = (e @ values) / l[:, None]
    lse[rows] = m + np.log(l)
    return out, lse


def attention_weights(q_row: np.ndarray, keys: np.ndarray, scale: float) -> np.ndarray:
    """The softmax weights of one query row over all its keys (for invariant checks)."""
    z = float(scale) * (_f64(keys) @ _f64(q_row))
    e = np.exp(z - z.max())
    return e / e.sum()


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale):
    """One query token per sequence: ``q`` [S, H, D] over pages [nb, bs, G, D].

    Returns ``(out [S, H, D], lse [S, H])``.  The query is the sequence's
    last cached position, so it sees all ``seq_lens[s]`` tokens.
    """
    q = _f64(q)
    k_cache = _arr(k_cache)
    v_cache = _arr(v_cache)
    S, H, D = q.shape
    bs, G = k_cache.shape[1], k_cache.shape[2]
    if H % G:
        raise ValueError("q heads must be a multiple of kv heads")
    r = H // G
    out = np.zeros((S, H, v_cache.shape[3]), dtype=np.float64)
    lse = np.full((S, H), NEG_INF, dtype=np.float64)
    bt = _ints(block_table)
    for s in range(S):
        L = int(_ints(seq_lens)[s])
        if L <= 0:
            continue
        for g in range(G):
            K = _f64(gather_tokens(k_cache[:, :, g], bt[s], L, bs))
            V = _f64(gather_tokens(v_cache[:, :, g], bt[s], L, bs))
            heads = slice(g * r, (g + 1) * r)
            o, l = softmax_attention(q[s, heads], K, V, scale, np.full(r, L))
            out[s, heads] = o
            lse[s, heads] = l
    return out, lse


def paged_prefill(q, cu_q_lens, k_cache, v_cache, block_table, seq_lens, scale):
    """Chunked prefill: sequence ``s`` queries its last ``q_len`` cached tokens.

    ``q`` [T, H, D] packs the sequences' query rows back to back
    (``cu_q_lens`` [S + 1]).  Row ``i`` of the chunk sits at position
    ``L - q_len + i`` and sees keys ``0 .. L - q_len + i`` (causal inside the
    chunk, everything in the cached prefix).  Returns ``(out [T, H, D],
    lse [T, H])``.
    """
    q = _f64(q)
    k_cache = _arr(k_cache)
    v_cache = _arr(v_cache)
    T, H, D = q.shape
    bs, G = k_cache.shape[1], k_cache.shape[2]
    if H % G:
        raise ValueError("q heads must be a multiple of kv heads")
    r = H // G
    cu = _ints(cu_q_lens).astype(np.int64)
    bt = _ints(block_table)
    out = np.zeros((T, H, v_cache.shape[3]), dtype=np.float64)
    lse = np.full((T, H), NEG_INF, dtype=np.float64)
    for s in range(len(cu) - 1):
        q0, q1 = int(cu[s]), int(cu[s + 1])
        q_len = q1 - q0
        L = int(_ints(seq_lens)[s])
        if q_len <= 0:
            continue
        if q_len > L:
            raise ValueError("a sequence queries more tokens than it holds")
        visible = (L - q_len) + np.arange(q_len) + 1
        for g in range(G):
            K = _f64(gather_tokens(k_cache[:, :, g], bt[s], L, bs))
            V = _f64(gather_tokens(v_cache[:, :, g], bt[s], L, bs))
            for h in range(g * r, (g + 1) * r):
                o, l = softmax_attention(q[q0:q1, h], K, V, scale, visible)
                out[q0:q1, h] = o
                lse[q0:q1, h] = l
    return out, lse


def paged_prefill_rows(q, cu_q_lens, k_cache, v_cache, block_table, seq_lens, scale, rows):
    """The same as :func:`paged_prefill` for the listed ``(token, head)`` rows only.

    Used to check sampled outputs of full-size workloads.  Returns
    ``(out [n, D], lse [n])`` in the order of ``rows``.
    """
    q = _arr(q)
    k_cache = _arr(k_cache)
    v_cache = _arr(v_cache)
    H = q.shape[1]
    bs, G = k_cache.shape[1], k_cache.shape[2]
    r = H // G
    cu = _ints(cu_q_lens).astype(np.int64)
    bt = _ints(block_table)
    out = np.zeros((len(rows), v_cache.shape[3]))
    lse = np.full(len(rows), NEG_INF)
    for n, (tok, h) in enumerate(rows):
        s = int(np.searchsorted(cu, tok, side="right") - 1)
        q_len = int(cu[s + 1] - cu[s])
        L = int(_ints(seq_lens)[s])
        i = int(tok - cu[s])
        g = h // r
        K = _f64(gather_tokens(k_cache[:, :, g], bt[s], L, bs))
        V = _f64(gather_tokens(v_cache[:, :, g], bt[s], L, bs))
        o, l = softmax_attention(_f64(q[tok, h])[None], K, V, scale, np.array([L - q_len + i + 1]))
        out[n] = o[0]
        lse[n] = l[0]
    return out, lse


def mla_decode(q, kv_cache, block_table, seq_lens, scale, d_latent=512):
    """MLA decode: every q head attends over one shared latent page pool.

    ``q`` [S, H, d_latent + d_rope]; ``kv_cache`` [nb, bs, d_latent + d_rope].
    The key is the full latent+rope row, the value its first ``d_latent``
    columns.  Returns ``(out [S, H, d_latent], lse [S, H])``.
    """
    q = _f64(q)
    kv_cache = _arr(kv_cache)
    S, H, dq = q.shape
    bs = kv_cache.shape[1]
    bt = _ints(block_table)
    out = np.zeros((S, H, d_latent), dtype=np.float64)
    lse = np.full((S, H), NEG_INF, dtype=np.float64)
    for s in range(S):
        L = int(_ints(seq_lens)[s])
        if L <= 0:
            continue
        rows = _f64(gather_tokens(kv_cache, bt[s], L, bs))   # [L, dq]
        o, l = softmax_attention(q[s], rows, rows[:, :d_latent], scale, np.full(H, L))
        out[s] = o
        lse[s] = l
    return out, lse


def split_partials(q_rows, keys, values, scale, partition_size):
    """Step 6, first half: softmax over each ``partition_size``-token partition.

    Returns ``(o_parts [P, n, Dv], lse_parts [P, n])``; each partial output
    is normalised within its partition.
    """
    L = keys.shape[0]
    n = q_rows.shape[0]
    P = max(1, -(-L // partition_size))
    o_parts = np.zeros((P, n, values.shape[1]))
    lse_parts = np.full((P, n), NEG_INF)
    for p in range(P):
        lo, hi = p * partition_size, min(L, (p + 1) * partition_size)
        if hi <= lo:
            continue
        o, l = softmax_attention(q_rows, keys[lo:hi], values[lo:hi], scale, np.full(n, hi - lo))
        o_parts[p] = o
        lse_parts[p] = l
    return o_parts, lse_parts


def merge_states(o_parts, lse_parts):
    """Step 6, second half: the log-sum-exp merge of partial attention results.

    ``lse = m + ln sum_p exp(lse_p - m)`` with ``m = max_p lse_p``;
    ``out = sum_p exp(lse_p - lse) o_p``.  Partitions with ``lse_p = -inf``
    weigh nothing; if every partition is empty the result is ``(0, -inf)``.
    ``o_parts`` [P, ..., Dv], ``lse_parts`` [P, ...].
    """
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe[None]), 0.0)
    total = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), NEG_INF)
    coef = np.where(finite[None], w / np.where(finite, total, 1.0)[None], 0.0)
    # an empty partition's output is undefined (it was never written): skip it, don't multiply it by 0
    out = np.where(coef[..., None] > 0, coef[..., None] * o_parts, 0.0).sum(axis=0)
    return out, lse


def paged_decode_split(q, k_cache, v_cache, block_table, seq_lens, scale, partition_size):
    """Decode through split partials + merge (used to check merge == unsplit).

    Returns ``(out, lse, o_parts_list, lse_parts_list)`` where the lists are
    indexed ``[s][g]``.
    """
    q = _f64(q)
    k_cache = _arr(k_cache)
    v_cache = _arr(v_cache)
    S, H, D = q.shape
    bs, G = k_cache.shape[1], k_cache.shape[2]
    r = H // G
    bt = _ints(block_table)
    out = np.zeros((S, H, v_cache.shape[3]))
    lse = np.full((S, H), NEG_INF)
    for s in range(S):
        L = int(_ints(seq_lens)[s])
        if L <= 0:
            continue
        for g in range(G):
            K = _f64(gather_tokens(k_cache[:, :, g], bt[s], L, bs))
            V = _f64(gather_tokens(v_cache[:, :, g], bt[s], L, bs))
            heads = slice(g * r, (g + 1) * r)
            op, lp = split_partials(q[s, heads], K, V, scale, partition_size)
            o, l = merge_states(op, lp)
            out[s, heads] = o
            lse[s, heads] = l
    return out, lse
