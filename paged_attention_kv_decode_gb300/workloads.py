"""Seeded synthetic inputs for paged attention over a paged KV cache.

This module only draws inputs: sequence lengths, the physical placement of
KV pages in the block pool, and N(0, 1) query / key / value values, rounded
to the storage dtype.  It holds none of the attention arithmetic, so both the
CUDA path and the CPU oracle can consume its output without sharing any of
the method.

Layouts (the problem statement of the vLLM paged-attention plugins, e.g. the
vllm-metal article, section 4: the scheduler hands the kernels a block table
and per-sequence lengths):

* ``k_cache`` / ``v_cache``: ``[num_blocks, block_size, kv_heads, head_dim]``.
* MLA ``kv_cache``: ``[num_blocks, block_size, d_latent + d_rope]`` (one latent
  head; latent columns first, rope columns last).
* ``block_table``: int32 ``[num_seqs, max_blocks]``; logical page ``j`` of
  sequence ``s`` lives in physical block ``block_table[s, j]``; unused slots
  hold -1.
* ``seq_lens``: int32 ``[num_seqs]``, the number of cached tokens per sequence,
  including the tokens being queried.

Draw order for every case: lengths, then the block permutation, then q, then
the K pool, then the V pool (float32 N(0, 1), rounded to the storage dtype by
torch).  ``poison=True`` overwrites, after the draw, every pool entry the
method must not read (blocks no sequence owns, and the tail slots of each
sequence's last page) with NaN, so that a read through a wrong index shows up.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

F32 = torch.float32
BF16 = torch.bfloat16

# Values are drawn in chunks of this many blocks so that the float32 staging
# buffer stays small for the multi-GB pools.
_CHUNK_ELEMS = 1 << 25


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(rng: np.random.Generator, shape: Sequence[int], dtype: torch.dtype) -> torch.Tensor:
    """N(0, 1) float32 draws rounded (RNE, by torch) to ``dtype``, drawn chunkwise."""
    shape = tuple(int(x) for x in shape)
    out = torch.empty(shape, dtype=dtype)
    if out.numel() == 0:
        return out
    flat = out.view(-1)
    n = flat.numel()
    step = _CHUNK_ELEMS
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        chunk = rng.standard_normal(hi - lo, dtype=np.float32)
        flat[lo:hi] = torch.from_numpy(chunk).to(dtype)
    return out


def _deal_blocks(rng: np.random.Generator, pages_per_seq: np.ndarray, num_blocks: int):
    """One random permutation of the pool, dealt out to the sequences in order."""
    total = int(pages_per_seq.sum())
    assert total <= num_blocks, (total, num_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(1, int(pages_per_seq.max()) if len(pages_per_seq) else 1)
    table = np.full((len(pages_per_seq), max_blocks), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(pages_per_seq):
        table[s, :n] = perm[off:off + n]
        off += n
    return torch.from_numpy(table)


def _poison_pool(pool: torch.Tensor, block_table: torch.Tensor, seq_lens: np.ndarray, bs: int):
    """NaN wherever no sequence holds a token: unowned blocks and page tails."""
    nb = pool.shape[0]
    owned = torch.zeros(nb, dtype=torch.bool)
    bt = block_table.numpy()
    for s, L in enumerate(seq_lens):
        n = -(-int(L) // bs)
        if n == 0:
            continue
        ids = bt[s, :n]
        owned[torch.from_numpy(ids.astype(np.int64))] = True
        tail = int(L) - (n - 1) * bs
        if tail < bs:
            pool[int(ids[n - 1]), tail:] = float("nan")
    pool[~owned] = float("nan")


@dataclasses.dataclass
class DecodeCase:
    """One query token per sequence over a paged K/V cache (GQA)."""
    name: str
    q: torch.Tensor            # [S, H, D]
    k_cache: torch.Tensor      # [nb, bs, G, D]
    v_cache: torch.Tensor      # [nb, bs, G, D]
    block_table: torch.Tensor  # int32 [S, max_blocks]
    seq_lens: torch.Tensor     # int32 [S]
    scale: float
    partition_size: int = 0    # 0: one pass over the whole sequence

    @property
    def S(self): return self.q.shape[0]
    @property
    def H(self): return self.q.shape[1]
    @property
    def D(self): return self.q.shape[2]
    @property
    def G(self): return self.k_cache.shape[2]
    @property
    def bs(self): return self.k_cache.shape[1]
    @property
    def num_blocks(self): return self.k_cache.shape[0]
    @property
    def max_blocks(self): return self.block_table.shape[1]
    @property
    def dtype(self): return self.q.dtype
    @property
    def max_seq_len(self): return int(self.seq_lens.max()) if self.S else 0


@dataclasses.dataclass
class PrefillCase:
    """Query chunks (``q_len`` tokens per sequence, packed) over prefix + chunk pages."""
    name: str
    q: torch.Tensor            # [T, H, D], T = sum of q_lens
    cu_q_lens: torch.Tensor    # int32 [S + 1]
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor     # int32 [S]: cached prefix + q_len
    scale: float

    @property
    def S(self): return self.seq_lens.shape[0]
    @property
    def T(self): return self.q.shape[0]
    @property
    def H(self): return self.q.shape[1]
    @property
    def D(self): return self.q.shape[2]
    @property
    def G(self): return self.k_cache.shape[2]
    @property
    def bs(self): return self.k_cache.shape[1]
    @property
    def num_blocks(self): return self.k_cache.shape[0]
    @property
    def max_blocks(self): return self.block_table.shape[1]
    @property
    def dtype(self): return self.q.dtype
    @property
    def q_lens(self): return (self.cu_q_lens[1:] - self.cu_q_lens[:-1])
    @property
    def max_q_len(self): return int(self.q_lens.max()) if self.S else 0
    @property
    def max_seq_len(self): return int(self.seq_lens.max()) if self.S else 0


@dataclasses.dataclass
class MLACase:
    """Multi-head latent attention decode over one shared latent page pool."""
    name: str
    q: torch.Tensor            # [S, H, d_latent + d_rope]
    kv_cache: torch.Tensor     # [nb, bs, d_latent + d_rope]
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    scale: float
    d_latent: int = 512
    d_rope: int = 64
    partition_size: int = 0

    @property
    def S(self): return self.q.shape[0]
    @property
    def H(self): return self.q.shape[1]
    @property
    def bs(self): return self.kv_cache.shape[1]
    @property
    def num_blocks(self): return self.kv_cache.shape[0]
    @property
    def max_blocks(self): return self.block_table.shape[1]
    @property
    def max_seq_len(self): return int(self.seq_lens.max()) if self.S else 0


def _pages(seq_lens: np.ndarray, bs: int) -> np.ndarray:
    return np.array([-(-int(L) // bs) for L in seq_lens], dtype=np.int64)


def make_decode_case(seed: int, seq_lens: Sequence[int], H: int, G: int, D: int, bs: int,
                     dtype: torch.dtype, scale: Optional[float] = None, num_blocks: Optional[int] = None,
                     extra_blocks: int = 0, poison: bool = False, partition_size: int = 0,
                     name: str = "decode", rng: Optional[np.random.Generator] = None) -> DecodeCase:
    """A decode batch with the given lengths; the pool is exactly the pages needed plus ``extra_blocks``."""
    rng = rng if rng is not None else _rng(seed)
    lens = np.asarray(seq_lens, dtype=np.int64)
    pages = _pages(lens, bs)
    nb = int(num_blocks) if num_blocks is not None else int(pages.sum()) + int(extra_blocks)
    nb = max(nb, 1)
    block_table = _deal_blocks(rng, pages, nb)
    S = len(lens)
    q = _normal(rng, (S, H, D), dtype)
    k = _normal(rng, (nb, bs, G, D), dtype)
    v = _normal(rng, (nb, bs, G, D), dtype)
    if poison:
        _poison_pool(k, block_table, lens, bs)
        _poison_pool(v, block_table, lens, bs)
    return DecodeCase(name=name, q=q, k_cache=k, v_cache=v, block_table=block_table,
                      seq_lens=torch.from_numpy(lens.astype(np.int32)),
                      scale=float(scale) if scale is not None else 1.0 / math.sqrt(D),
                      partition_size=partition_size)


def make_prefill_case(seed: int, prefix_lens: Sequence[int], q_lens: Sequence[int], H: int, G: int, D: int,
                      bs: int, dtype: torch.dtype, scale: Optional[float] = None, extra_blocks: int = 0,
                      poison: bool = False, name: str = "prefill",
                      rng: Optional[np.random.Generator] = None) -> PrefillCase:
    """Each sequence holds ``prefix + q_len`` cached tokens; its last ``q_len`` are queried."""
    rng = rng if rng is not None else _rng(seed)
    prefix = np.asarray(prefix_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    assert prefix.shape == ql.shape
    lens = prefix + ql
    pages = _pages(lens, bs)
    nb = max(1, int(pages.sum()) + int(extra_blocks))
    block_table = _deal_blocks(rng, pages, nb)
    T = int(ql.sum())
    q = _normal(rng, (T, H, D), dtype)
    k = _normal(rng, (nb, bs, G, D), dtype)
    v = _normal(rng, (nb, bs, G, D), dtype)
    if poison:
        _poison_pool(k, block_table, lens, bs)
        _poison_pool(v, block_table, lens, bs)
    cu = np.zeros(len(ql) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    return PrefillCase(name=name, q=q, cu_q_lens=torch.from_numpy(cu), k_cache=k, v_cache=v,
                       block_table=block_table, seq_lens=torch.from_numpy(lens.astype(np.int32)),
                       scale=float(scale) if scale is not None else 1.0 / math.sqrt(D))


def make_mla_case(seed: int, seq_lens: Sequence[int], H: int, bs: int, d_latent: int = 512, d_rope: int = 64,
                  scale: Optional[float] = None, extra_blocks: int = 0, poison: bool = False,
                  partition_size: int = 0, name: str = "mla",
                  rng: Optional[np.random.Generator] = None) -> MLACase:
    rng = rng if rng is not None else _rng(seed)
    lens = np.asarray(seq_lens, dtype=np.int64)
    pages = _pages(lens, bs)
    nb = max(1, int(pages.sum()) + int(extra_blocks))
    block_table = _deal_blocks(rng, pages, nb)
    S = len(lens)
    dq = d_latent + d_rope
    q = _normal(rng, (S, H, dq), BF16)
    kv = _normal(rng, (nb, bs, dq), BF16)
    if poison:
        _poison_pool(kv, block_table, lens, bs)
    return MLACase(name=name, q=q, kv_cache=kv, block_table=block_table,
                   seq_lens=torch.from_numpy(lens.astype(np.int32)),
                   scale=float(scale) if scale is not None else 1.0 / math.sqrt(192.0),
                   d_latent=d_latent, d_rope=d_rope, partition_size=partition_size)


# ---------------------------------------------------------------------------
# The five workloads.  Each builder takes a ``shrink`` divisor for the
# sequence count and the length range so that parity tests can run the same
# recipe at sizes the oracle finishes in seconds.
# ---------------------------------------------------------------------------

def _uniform_lens(rng, n, lo, hi):
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def config1_tiny_decode(poison: bool = False) -> DecodeCase:
    """4 seqs, lengths U[1, 64], 4 q heads / 1 kv head, head_dim 64, block 16, 32 permuted blocks, fp32."""
    rng = _rng(1001)
    lens = _uniform_lens(rng, 4, 1, 64)
    return make_decode_case(1001, lens, H=4, G=1, D=64, bs=16, dtype=F32, scale=1.0 / 8.0,
                            num_blocks=32, poison=poison, name="c1_tiny_decode_fp32", rng=rng)


def config2_batched_decode(poison: bool = False, num_seqs: int = 64, len_lo: int = 512, len_hi: int = 4096,
                           partition_size: int = 0, extra_blocks: int = 0) -> DecodeCase:
    """64 seqs, lengths U[512, 4096], 32 q / 8 kv heads, head_dim 128, block 16, bf16."""
    rng = _rng(1002)
    lens = _uniform_lens(rng, num_seqs, len_lo, len_hi)
    return make_decode_case(1002, lens, H=32, G=8, D=128, bs=16, dtype=BF16, poison=poison,
                            partition_size=partition_size, extra_blocks=extra_blocks,
                            name="c2_batched_decode_bf16", rng=rng)


def config3_long_split_decode(poison: bool = False, num_seqs: int = 8, len_lo: int = 32768,
                              len_hi: int = 131072, partition_size: int = 512,
                              extra_blocks: int = 0) -> DecodeCase:
    """8 seqs, lengths U[32768, 131072], 32 q / 8 kv heads, head_dim 128, block 16, 512-token partitions."""
    rng = _rng(1003)
    lens = _uniform_lens(rng, num_seqs, len_lo, len_hi)
    return make_decode_case(1003, lens, H=32, G=8, D=128, bs=16, dtype=BF16, poison=poison,
                            partition_size=partition_size, extra_blocks=extra_blocks,
                            name="c3_long_split_decode_bf16", rng=rng)


def config4_chunked_prefill(poison: bool = False, num_chunks: int = 16, chunk: int = 512,
                            prefix_hi: int = 4096, num_decodes: int = 48, dec_lo: int = 512,
                            dec_hi: int = 4096, extra_blocks: int = 0) -> PrefillCase:
    """16 chunks of 512 over prefixes U[0, 4096], mixed with 48 decodes of U[512, 4096], shuffled."""
    rng = _rng(1004)
    prefix_c = _uniform_lens(rng, num_chunks, 0, prefix_hi)
    dec_lens = _uniform_lens(rng, num_decodes, dec_lo, dec_hi)
    prefix = np.concatenate([prefix_c, dec_lens - 1])
    ql = np.concatenate([np.full(num_chunks, chunk, dtype=np.int64), np.ones(num_decodes, dtype=np.int64)])
    order = rng.permutation(len(ql))
    return make_prefill_case(1004, prefix[order], ql[order], H=32, G=8, D=128, bs=16, dtype=BF16,
                             poison=poison, extra_blocks=extra_blocks, name="c4_chunked_prefill_bf16", rng=rng)


def mla_lengths(rng, n, median=1024, sigma=1.0, cap=8192):
    """Lognormal lengths: round(exp(N(ln median, sigma))), clamped to [1, cap]."""
    x = np.exp(rng.normal(math.log(median), sigma, size=n))
    return np.clip(np.rint(x), 1, cap).astype(np.int64)


def config5_mla_decode(poison: bool = False, num_seqs: int = 128, median: int = 1024, cap: int = 8192,
                       partition_size: int = 0, extra_blocks: int = 0) -> MLACase:
    """128 seqs, lognormal lengths (median 1024, cap 8192), 128 heads, latent 512 + rope 64, block 64."""
    rng = _rng(1005)
    lens = mla_lengths(rng, num_seqs, median=median, cap=cap)
    return make_mla_case(1005, lens, H=128, bs=64, poison=poison, partition_size=partition_size,
                         extra_blocks=extra_blocks, name="c5_mla_decode_bf16", rng=rng)


class PrefixCase:
    """Prompts for the prefix-cache lookup: tokens, offsets and a free-page stack.

    ``tokens`` int32 ``[T]`` (the prompts concatenated), ``cu_tokens`` /
    ``cu_pages`` int32 ``[S + 1]`` (token and full-page offsets), ``free_stack``
    int32 ``[num_pages]`` (a seeded permutation of the page ids, top at the end).
    """

    def __init__(self, name, tokens, cu_tokens, block_size, num_pages, free_stack):
        self.name = name
        self.tokens = tokens
        self.cu_tokens = cu_tokens
        self.block_size = block_size
        lens = np.diff(cu_tokens)
        self.cu_pages = np.concatenate([[0], np.cumsum(lens // block_size)]).astype(np.int32)
        self.total_pages = int(self.cu_pages[-1])
        self.num_pages = num_pages
        self.free_stack = free_stack

    @property
    def num_seqs(self) -> int:
        return len(self.cu_tokens) - 1

    @property
    def num_tokens(self) -> int:
        return int(self.cu_tokens[-1])


def make_prefix_case(seed: int, num_seqs: int, num_prefixes: int, prefix_lo: int, prefix_hi: int, suffix_lo: int,
                     suffix_hi: int, bs: int, num_pages: int, vocab: int = 32000, name: str = "prefix") -> PrefixCase:
    """Each prompt = one of ``num_prefixes`` shared system prompts (lengths uniform in
    [prefix_lo, prefix_hi]) followed by its own suffix (uniform in [suffix_lo, suffix_hi]);
    token ids uniform in [0, vocab).  Draw order: prefix lengths, prefix tokens, the prefix
    choice per prompt, suffix lengths, suffix tokens, then the free-stack permutation."""
    rng = _rng(seed)
    plens = rng.integers(prefix_lo, prefix_hi + 1, size=num_prefixes)
    prefixes = [rng.integers(0, vocab, size=int(n), dtype=np.int64).astype(np.int32) for n in plens]
    choice = rng.integers(0, num_prefixes, size=num_seqs)
    slens = rng.integers(suffix_lo, suffix_hi + 1, size=num_seqs)
    parts = []
    for s in range(num_seqs):
        parts.append(prefixes[choice[s]])
        parts.append(rng.integers(0, vocab, size=int(slens[s]), dtype=np.int64).astype(np.int32))
    tokens = np.concatenate(parts) if parts else np.zeros(0, np.int32)
    lens = plens[choice] + slens
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    stack = rng.permutation(num_pages).astype(np.int32)
    return PrefixCase(name, tokens, cu, bs, num_pages, stack)


def prefix_workload(num_seqs: int = 4096) -> PrefixCase:
    """4096 prompts of 640-768 tokens sharing 16 system prompts of 576-640 tokens, block 16,
    a pool of 262144 pages (the repeated-prompt shape of the vllm-metis status report)."""
    return make_prefix_case(1006, num_seqs, 16, 576, 640, 32, 160, 16, 262144, name="prefix_lookup_4096x700")


CONFIGS = {
    "c1": config1_tiny_decode,
    "c2": config2_batched_decode,
    "c3": config3_long_split_decode,
    "c4": config4_chunked_prefill,
    "c5": config5_mla_decode,
}
