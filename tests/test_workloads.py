"""Host-side checks of the seeded workload generator (no GPU)."""

import numpy as np
import torch

from paged_attention_kv_decode_gb300 import workloads as wl


def _check_table(bt, seq_lens, bs, nb):
    bt = bt.numpy()
    used = []
    for s, L in enumerate(seq_lens.numpy()):
        n = -(-int(L) // bs)
        assert (bt[s, :n] >= 0).all() and (bt[s, :n] < nb).all()
        assert (bt[s, n:] == -1).all()
        used.extend(bt[s, :n].tolist())
    assert len(used) == len(set(used)), "a physical block is dealt twice"


def test_config1_shape_and_table():
    c = wl.config1_tiny_decode()
    assert c.q.shape == (4, 4, 64) and c.q.dtype == torch.float32
    assert c.k_cache.shape == (32, 16, 1, 64)
    assert ((c.seq_lens >= 1) & (c.seq_lens <= 64)).all()
    _check_table(c.block_table, c.seq_lens, 16, 32)
    assert abs(c.scale - 0.125) < 1e-15


def test_seeded_and_reproducible():
    a = wl.config1_tiny_decode()
    b = wl.config1_tiny_decode()
    assert torch.equal(a.q, b.q) and torch.equal(a.k_cache, b.k_cache) and torch.equal(a.block_table, b.block_table)


def test_config2_recipe_small():
    c = wl.config2_batched_decode(num_seqs=6, len_lo=17, len_hi=100)
    assert c.q.shape == (6, 32, 128) and c.q.dtype == torch.bfloat16
    assert c.k_cache.shape[1:] == (16, 8, 128)
    pages = sum(-(-int(L) // 16) for L in c.seq_lens)
    assert c.num_blocks == pages
    _check_table(c.block_table, c.seq_lens, 16, c.num_blocks)


def test_config4_mix_small():
    c = wl.config4_chunked_prefill(num_chunks=3, chunk=40, prefix_hi=50, num_decodes=5, dec_lo=10, dec_hi=30)
    ql = c.q_lens.numpy()
    assert sorted(ql.tolist()) == [1] * 5 + [40] * 3
    assert c.T == 3 * 40 + 5
    assert (c.seq_lens.numpy() >= ql).all()
    _check_table(c.block_table, c.seq_lens, 16, c.num_blocks)


def test_config5_lognormal_lengths():
    rng = np.random.Generator(np.random.PCG64(0))
    lens = wl.mla_lengths(rng, 20000)
    assert lens.min() >= 1 and lens.max() <= 8192
    assert abs(np.median(lens) - 1024) < 40
    c = wl.config5_mla_decode(num_seqs=4, median=50, cap=200)
    assert c.q.shape == (4, 128, 576) and c.kv_cache.shape[1:] == (64, 576)


def test_poison_marks_only_unread_entries():
    c = wl.make_decode_case(3, [5, 16, 17], H=2, G=1, D=4, bs=16, dtype=torch.float32, extra_blocks=2,
                            poison=True)
    bt = c.block_table.numpy()
    k = c.k_cache.numpy()
    for s, L in enumerate(c.seq_lens.numpy()):
        for t in range(int(L)):
            assert np.isfinite(k[bt[s, t // 16], t % 16]).all()
    assert np.isnan(k).sum() == (2 * 16 + 11 + 15) * 4
