"""Pins of the KV-cache-write oracle (no GPU).

Each pin ties the oracle to something other than itself: a row-by-row brute
force written independently, the attention oracle's block-table gather (the
write followed by the read must return the contiguous rows), and the
attention result over contiguous tensors.
"""
import numpy as np
import pytest
import torch

import oracle


def _pool(nb, bs, G, D, dtype):
    return torch.full((nb, bs, G, D), float("nan"), dtype=dtype)


def test_brute_force_tiny():
    nb, bs, G, D = 3, 4, 2, 2
    key = torch.arange(3 * G * D, dtype=torch.float32).reshape(3, G, D)
    value = -key
    kc, vc = oracle.reshape_and_cache(key, value, torch.zeros(nb, bs, G, D), torch.zeros(nb, bs, G, D),
                                      [5, -1, 11])
    want_k = torch.zeros(nb, bs, G, D)
    want_k[1, 1] = key[0]          # slot 5 = block 1, offset 1
    want_k[2, 3] = key[2]          # slot 11 = block 2, offset 3
    assert torch.equal(kc, want_k)
    assert torch.equal(vc, -want_k)


def test_inputs_untouched_and_padding_skipped():
    k0 = torch.randn(2, 4, 1, 8)
    v0 = torch.randn(2, 4, 1, 8)
    key = torch.randn(3, 1, 8)
    kc, vc = oracle.reshape_and_cache(key, key, k0, v0, torch.tensor([-1, -1, -1]))
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
    kc, _ = oracle.reshape_and_cache(key, key, k0, v0, torch.tensor([0, -5, 7]))
    assert not torch.equal(kc, k0) and torch.equal(k0, k0.clone())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bs", [16, 64])
def test_write_then_gather_round_trip(dtype, bs):
    """Write a sequence's contiguous rows through a permuted block table, read them
    back with the attention oracle's gather: bitwise the same rows, the rest NaN."""
    rng = np.random.default_rng(3)
    L, G, D = 150, 4, 16
    n_pages = -(-L // bs)
    nb = n_pages + 5
    table = rng.permutation(nb)[:n_pages]
    K = torch.randn(L, G, D).to(dtype)
    V = torch.randn(L, G, D).to(dtype)
    t = np.arange(L)
    slots = torch.from_numpy(table[t // bs] * bs + t % bs)
    kc, vc = oracle.reshape_and_cache(K, V, _pool(nb, bs, G, D, dtype), _pool(nb, bs, G, D, dtype), slots)
    for g in range(G):
        assert torch.equal(oracle.gather_tokens(kc[:, :, g], table, L, bs), K[:, g])
        assert torch.equal(oracle.gather_tokens(vc[:, :, g], table, L, bs), V[:, g])
    written = torch.zeros(nb * bs, dtype=torch.bool)
    written[slots] = True
    assert torch.isnan(kc.float().reshape(nb * bs, -1)[~written]).all()


def test_write_then_decode_equals_contiguous_attention():
    rng = np.random.default_rng(4)
    L, G, H, D, bs = 70, 2, 4, 32, 16
    nb = 9
    table = rng.permutation(nb)[: -(-L // bs)]
    K = torch.randn(L, G, D, dtype=torch.float64)
    V = torch.randn(L, G, D, dtype=torch.float64)
    q = torch.randn(1, H, D, dtype=torch.float64)
    t = np.arange(L)
    kc, vc = oracle.reshape_and_cache(K, V, torch.zeros(nb, bs, G, D, dtype=torch.float64),
                                      torch.zeros(nb, bs, G, D, dtype=torch.float64), table[t // bs] * bs + t % bs)
    bt = np.full((1, nb), -1)
    bt[0, : len(table)] = table
    out, _ = oracle.paged_decode(q, kc, vc, bt, np.array([L]), 0.2)
    r = H // G
    for h in range(H):
        o, _ = oracle.softmax_attention(q[0, h:h + 1].numpy(), K[:, h // r].numpy(), V[:, h // r].numpy(), 0.2,
                                        np.array([L]))
        np.testing.assert_allclose(out[0, h], o[0], rtol=1e-12, atol=1e-14)


def test_slot_past_pool_raises():
    with pytest.raises(IndexError):
        oracle.reshape_and_cache(torch.zeros(1, 1, 4), torch.zeros(1, 1, 4), torch.zeros(2, 4, 1, 4),
                                 torch.zeros(2, 4, 1, 4), [8])


def test_mla_write_brute_force_and_round_trip():
    nb, bs, dl, dr = 4, 16, 8, 4
    kv_c = torch.randn(20, dl).to(torch.bfloat16)
    k_pe = torch.randn(20, dr).to(torch.bfloat16)
    table = np.array([2, 0])
    t = np.arange(20)
    slots = table[t // bs] * bs + t % bs
    slots[3] = -1
    kc = oracle.mla_reshape_and_cache(kv_c, k_pe, torch.full((nb, bs, dl + dr), float("nan")).to(torch.bfloat16),
                                      torch.from_numpy(slots))
    rows = oracle.gather_tokens(kc, table, 20, bs)
    for n in range(20):
        if n == 3:
            assert torch.isnan(rows[n].float()).all()
        else:
            assert torch.equal(rows[n], torch.cat([kv_c[n], k_pe[n]]))
