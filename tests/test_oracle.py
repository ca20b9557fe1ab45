"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each pin is chosen so that a plausible mistake in the oracle fails it:

* a wrong page/slot convention or a wrong gather -> hand-worked block walk,
  contiguous brute force with the test's own scatter, poisoned pools;
* a dropped scale, wrong sign or transposed operand -> pure-Python brute
  force, two-key closed form, torch SDPA in float64;
* a wrong GQA head mapping -> torch SDPA with K/V repeated per group;
* top-left instead of bottom-right causal alignment -> prefill rows equal the
  matching rows of a full causal SDPA over the whole sequence, chunking
  invariance, q_len = 1 equals decode;
* natural log vs log2 in lse -> scipy.special.logsumexp;
* a wrong merge weight -> split-then-merge equals unsplit, closed forms.
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from paged_attention_kv_decode_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# test-side helpers: a scatter of contiguous K/V into pages, and a brute
# force attention in plain Python.  Neither calls the oracle.
# ---------------------------------------------------------------------------

def scatter_into_pages(seqs_kv, bs, rng, extra_blocks=3, fill=np.nan):
    """Place contiguous per-sequence rows ``[L, ...]`` into a fresh page pool."""
    pages = [-(-x.shape[0] // bs) for x in seqs_kv]
    nb = sum(pages) + extra_blocks
    perm = rng.permutation(nb)
    trail = seqs_kv[0].shape[1:]
    pool = np.full((nb, bs) + trail, fill)
    table = np.full((len(seqs_kv), max(1, max(pages))), -1, dtype=np.int32)
    off = 0
    for s, x in enumerate(seqs_kv):
        for j in range(pages[s]):
            blk = perm[off + j]
            table[s, j] = blk
            chunk = x[j * bs:(j + 1) * bs]
            pool[blk, :chunk.shape[0]] = chunk
        off += pages[s]
    return pool, table


def brute_attention(q, K, V, scale):
    """Softmax attention of one query over all keys, in plain Python floats."""
    z = [scale * sum(float(a) * float(b) for a, b in zip(q, k)) for k in K]
    m = max(z)
    e = [math.exp(x - m) for x in z]
    l = sum(e)
    out = [sum(e[t] * float(V[t][d]) for t in range(len(K))) / l for d in range(len(V[0]))]
    return out, m + math.log(l)


def sdpa_f64(q, k, v, scale, causal):
    """torch SDPA (math backend, float64) for q [Hq, Lq, D], k/v [Hq, Lk, D]."""
    with torch.no_grad():
        return torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
            is_causal=causal, scale=scale)[0].numpy()


# ---------------------------------------------------------------------------
# gather / block table
# ---------------------------------------------------------------------------

def test_gather_hand_worked_block_walk():
    # block b, slot j holds the value 10*b + j; table [2, 0], bs 2, 3 tokens:
    # token 0 -> block 2 slot 0, token 1 -> block 2 slot 1, token 2 -> block 0 slot 0.
    cache = np.array([[[0.0], [1.0]], [[10.0], [11.0]], [[20.0], [21.0]]])
    rows = oracle.gather_tokens(cache, np.array([2, 0, -1]), 3, 2)
    assert rows[:, 0].tolist() == [20.0, 21.0, 0.0]


def test_gather_rejects_out_of_pool_ids():
    cache = np.zeros((2, 4, 1))
    with pytest.raises(IndexError):
        oracle.gather_tokens(cache, np.array([0, 5]), 6, 4)


def test_gather_reads_only_valid_slots():
    cache = np.full((3, 4, 1), np.nan)
    cache[1, :2, 0] = [1.0, 2.0]
    rows = oracle.gather_tokens(cache, np.array([1, -1, -1]), 2, 4)
    assert rows[:, 0].tolist() == [1.0, 2.0]


# ---------------------------------------------------------------------------
# decode vs brute force on contiguous data
# ---------------------------------------------------------------------------

def _tiny_decode(seed, lens, H=4, G=2, D=8, bs=4, scale=0.37):
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((L, G, D)) for L in lens]
    V = [rng.standard_normal((L, G, D)) for L in lens]
    q = rng.standard_normal((len(lens), H, D))
    return rng, q, K, V, scale


def test_decode_matches_python_brute_force():
    lens = [1, 5, 9, 4]
    H, G, D, bs = 4, 2, 8, 4
    rng, q, K, V, scale = _tiny_decode(7, lens, H, G, D, bs)
    kc, table = scatter_into_pages(K, bs, rng)
    vc, table2 = scatter_into_pages(V, bs, np.random.default_rng(12345))
    # the two scatters used different permutations: rebuild V with K's table
    vc = np.full_like(kc, np.nan)
    for s, L in enumerate(lens):
        for t in range(L):
            vc[table[s, t // bs], t % bs] = V[s][t]
    out, lse = oracle.paged_decode(q, kc, vc, table, np.array(lens), scale)
    r = H // G
    for s, L in enumerate(lens):
        for h in range(H):
            g = h // r
            o_ref, l_ref = brute_attention(q[s, h], K[s][:, g], V[s][:, g], scale)
            np.testing.assert_allclose(out[s, h], o_ref, rtol=0, atol=1e-12)
            assert abs(lse[s, h] - l_ref) < 1e-12


def test_block_permutation_invariance_is_bitwise():
    lens = [3, 17, 33]
    bs = 4
    rng, q, K, V, scale = _tiny_decode(11, lens, bs=bs)
    kv = [np.concatenate([k, v], axis=-1) for k, v in zip(K, V)]
    outs = []
    for perm_seed in (1, 2, 3):
        pool, table = scatter_into_pages(kv, bs, np.random.default_rng(perm_seed), extra_blocks=5)
        kc, vc = pool[..., :8], pool[..., 8:]
        outs.append(oracle.paged_decode(q, kc, vc, table, np.array(lens), scale))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0])
        assert np.array_equal(l, outs[0][1])


def test_poisoned_pool_never_read():
    case = wl.config1_tiny_decode(poison=True)
    clean = wl.config1_tiny_decode(poison=False)
    o1, l1 = oracle.paged_decode(case.q.numpy(), case.k_cache.numpy(), case.v_cache.numpy(),
                                 case.block_table.numpy(), case.seq_lens.numpy(), case.scale)
    o2, l2 = oracle.paged_decode(clean.q.numpy(), clean.k_cache.numpy(), clean.v_cache.numpy(),
                                 clean.block_table.numpy(), clean.seq_lens.numpy(), clean.scale)
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # the poisoning really covers something
    assert torch.isnan(case.k_cache).any()


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_two_key_closed_form():
    # q = (1, 0), k0 = (1, 0), k1 = (0, 1), scale 1: weights e/(e+1), 1/(e+1).
    kc = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])          # [1 block, bs 2, G 1, D 2]
    vc = np.array([[[[1.0, 2.0]], [[3.0, 4.0]]]])
    q = np.array([[[1.0, 0.0]]])
    out, lse = oracle.paged_decode(q, kc, vc, np.array([[0]]), np.array([2]), 1.0)
    w0 = math.e / (math.e + 1.0)
    w1 = 1.0 / (math.e + 1.0)
    np.testing.assert_allclose(out[0, 0], [w0 * 1 + w1 * 3, w0 * 2 + w1 * 4], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - math.log(math.e + 1.0)) < 1e-15


def test_length_one_returns_its_value_row_exactly():
    rng = np.random.default_rng(3)
    kc = rng.standard_normal((4, 16, 2, 8))
    vc = rng.standard_normal((4, 16, 2, 8))
    q = rng.standard_normal((2, 4, 8))
    table = np.array([[2, -1], [0, -1]], dtype=np.int32)
    out, _ = oracle.paged_decode(q, kc, vc, table, np.array([1, 1]), 0.5)
    for s, blk in ((0, 2), (1, 0)):
        for h in range(4):
            assert np.array_equal(out[s, h], vc[blk, 0, h // 2])


@pytest.mark.parametrize("mode", ["identical_keys", "zero_scale"])
def test_uniform_weights_give_mean_of_values(mode):
    rng = np.random.default_rng(5)
    L, bs = 37, 16
    kc = rng.standard_normal((3, bs, 1, 8))
    vc = rng.standard_normal((3, bs, 1, 8))
    if mode == "identical_keys":
        kc[:] = rng.standard_normal(8)
        scale = 0.9
    else:
        scale = 0.0
    q = rng.standard_normal((1, 2, 8))
    table = np.array([[1, 2, 0]], dtype=np.int32)
    out, lse = oracle.paged_decode(q, kc, vc, table, np.array([L]), scale)
    rows = [vc[table[0, t // bs], t % bs, 0] for t in range(L)]
    np.testing.assert_allclose(out[0, 0], np.mean(rows, axis=0), rtol=1e-14, atol=1e-14)
    if mode == "zero_scale":
        assert abs(lse[0, 0] - math.log(L)) < 1e-14


def test_weights_sum_to_one():
    rng = np.random.default_rng(9)
    kc = rng.standard_normal((5, 16, 2, 16)) * 3
    vc = np.ones((5, 16, 2, 16))
    q = rng.standard_normal((3, 4, 16))
    table = np.array([[0, 1, 2, 3, 4]] * 3, dtype=np.int32)
    out, _ = oracle.paged_decode(q, kc, vc, table, np.array([80, 17, 2]), 0.25)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-15)


def test_attention_weights_two_key_closed_form():
    # two keys whose scaled scores differ by d: the weights are the logistic
    # function of d, 1 / (1 + e^-d) and 1 / (1 + e^d)
    q = np.array([0.5, -1.0, 2.0])
    keys = np.array([[1.0, 0.0, 0.5], [0.0, 1.0, -0.5]])
    scale = 0.7
    d = scale * ((0.5 * 1.0 + 2.0 * 0.5) - (-1.0 * 1.0 + 2.0 * -0.5))   # scale * (z0 - z1), worked by hand
    w = oracle.attention_weights(q, keys, scale)
    assert w.shape == (2,)
    assert abs(w[0] - 1.0 / (1.0 + math.exp(-d))) < 1e-15
    assert abs(w[1] - 1.0 / (1.0 + math.exp(d))) < 1e-15


def test_attention_weights_match_python_brute_force():
    # sum to 1, non-negative, and equal to exp(z_t) / sum exp(z) evaluated in
    # plain Python floats; large scores (|z| ~ 300) would overflow an
    # unshifted exponential, so the brute force shifts by its own maximum
    rng = np.random.default_rng(29)
    for L, scale in ((1, 0.3), (5, 1.0), (40, 0.125), (17, 30.0)):
        q = rng.standard_normal(8)
        keys = rng.standard_normal((L, 8))
        w = oracle.attention_weights(q, keys, scale)
        z = [scale * sum(float(a) * float(b) for a, b in zip(q, k)) for k in keys]
        m = max(z)
        e = [math.exp(x - m) for x in z]
        ref = [x / sum(e) for x in e]
        assert (w >= 0).all()
        assert abs(w.sum() - 1.0) < 1e-14
        np.testing.assert_allclose(w, ref, rtol=1e-13, atol=1e-300)


def test_attention_weights_are_the_decode_weights():
    # the weighted sum of the value rows with these weights is the decode output
    # (a dropped scale or a transposed product in either would break it)
    rng = np.random.default_rng(31)
    L, bs, D = 45, 16, 16
    kc = rng.standard_normal((3, bs, 1, D))
    vc = rng.standard_normal((3, bs, 1, D))
    q = rng.standard_normal((1, 1, D))
    table = np.array([[2, 0, 1]], dtype=np.int32)
    out, _ = oracle.paged_decode(q, kc, vc, table, np.array([L]), 0.4)
    K = np.stack([kc[table[0, t // bs], t % bs, 0] for t in range(L)])
    V = np.stack([vc[table[0, t // bs], t % bs, 0] for t in range(L)])
    w = oracle.attention_weights(q[0, 0], K, 0.4)
    np.testing.assert_allclose(w @ V, out[0, 0], rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(13)
    kc = rng.standard_normal((2, 16, 1, 8)) * 0.01
    vc = rng.standard_normal((2, 16, 1, 8))
    q = np.zeros((1, 1, 8))
    q[0, 0, 3] = 1.0
    kc[1, 5, 0, 3] = 1e4                    # token 16 + 5 = 21 dominates by ~1e4
    out, _ = oracle.paged_decode(q, kc, vc, np.array([[0, 1]]), np.array([30]), 1.0)
    np.testing.assert_allclose(out[0, 0], vc[1, 5, 0], rtol=0, atol=1e-12)


def test_lse_equals_scipy_logsumexp():
    rng = np.random.default_rng(21)
    lens = [1, 7, 40]
    H, G, D, bs = 6, 3, 16, 8
    rng2, q, K, V, scale = _tiny_decode(21, lens, H, G, D, bs, scale=0.3)
    kv = [np.concatenate([k, v], -1) for k, v in zip(K, V)]
    pool, table = scatter_into_pages(kv, bs, rng)
    _, lse = oracle.paged_decode(q, pool[..., :D], pool[..., D:], table, np.array(lens), scale)
    for s, L in enumerate(lens):
        for h in range(H):
            z = scale * (K[s][:, h // 2] @ q[s, h])
            assert abs(lse[s, h] - logsumexp(z)) < 1e-12


# ---------------------------------------------------------------------------
# GQA mapping and the causal / chunked-prefill alignment, against torch SDPA
# ---------------------------------------------------------------------------

def test_prefill_prefix_zero_equals_causal_sdpa_with_gqa():
    rng = np.random.default_rng(31)
    H, G, D, bs = 8, 2, 16, 16
    lens = [45, 16, 1]
    K = [rng.standard_normal((L, G, D)) for L in lens]
    V = [rng.standard_normal((L, G, D)) for L in lens]
    kv = [np.concatenate([k, v], -1) for k, v in zip(K, V)]
    pool, table = scatter_into_pages(kv, bs, rng)
    q = rng.standard_normal((sum(lens), H, D))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    out, _ = oracle.paged_prefill(q, cu, pool[..., :D], pool[..., D:], table, np.array(lens), scale)
    for s, L in enumerate(lens):
        qs = q[cu[s]:cu[s + 1]].transpose(1, 0, 2)                      # [H, L, D]
        ks = np.repeat(K[s].transpose(1, 0, 2), H // G, axis=0)           # head h -> kv head h // (H/G)
        vs = np.repeat(V[s].transpose(1, 0, 2), H // G, axis=0)
        ref = sdpa_f64(qs.copy(), ks.copy(), vs.copy(), scale, causal=True)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]].transpose(1, 0, 2), ref, rtol=0, atol=1e-12)


def test_prefill_with_prefix_equals_tail_rows_of_full_causal_sdpa():
    rng = np.random.default_rng(37)
    H, G, D, bs = 4, 1, 16, 16
    L, prefix = 150, 87
    K = rng.standard_normal((L, G, D))
    V = rng.standard_normal((L, G, D))
    q_full = rng.standard_normal((L, H, D))
    pool, table = scatter_into_pages([np.concatenate([K, V], -1)], bs, rng)
    scale = 0.2
    cu = np.array([0, L - prefix], dtype=np.int32)
    out, _ = oracle.paged_prefill(q_full[prefix:], cu, pool[..., :D], pool[..., D:], table, np.array([L]), scale)
    ref = sdpa_f64(q_full.transpose(1, 0, 2).copy(), np.repeat(K.transpose(1, 0, 2), H, 0).copy(),
                   np.repeat(V.transpose(1, 0, 2), H, 0).copy(), scale, causal=True)
    np.testing.assert_allclose(out.transpose(1, 0, 2), ref[:, prefix:], rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 16, 64, 100])
def test_chunking_does_not_change_rows(chunk):
    rng = np.random.default_rng(41)
    H, G, D, bs = 4, 2, 8, 16
    L, prefix = 230, 30
    kc = rng.standard_normal((20, bs, G, D))
    vc = rng.standard_normal((20, bs, G, D))
    table = rng.permutation(20)[None, :].astype(np.int32)
    q = rng.standard_normal((L - prefix, H, D))
    whole, whole_lse = oracle.paged_prefill(q, np.array([0, L - prefix]), kc, vc, table, np.array([L]), 0.3)
    pos = prefix
    while pos < L:
        n = min(chunk, L - pos)
        part, part_lse = oracle.paged_prefill(q[pos - prefix:pos - prefix + n], np.array([0, n]), kc, vc, table,
                                              np.array([pos + n]), 0.3)
        np.testing.assert_allclose(part, whole[pos - prefix:pos - prefix + n], rtol=0, atol=1e-13)
        np.testing.assert_allclose(part_lse, whole_lse[pos - prefix:pos - prefix + n], rtol=0, atol=1e-13)
        pos += n


def test_prefill_single_token_equals_decode():
    case = wl.config1_tiny_decode()
    q = case.q.numpy()
    args = (case.k_cache.numpy(), case.v_cache.numpy(), case.block_table.numpy(), case.seq_lens.numpy())
    d_out, d_lse = oracle.paged_decode(q, *args, case.scale)
    cu = np.arange(case.S + 1, dtype=np.int32)
    p_out, p_lse = oracle.paged_prefill(q, cu, *args, case.scale)
    np.testing.assert_allclose(p_out, d_out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(p_lse, d_lse, rtol=0, atol=1e-14)


def test_prefill_rows_matches_prefill():
    case = wl.make_prefill_case(5, [0, 40, 7], [20, 9, 1], H=4, G=2, D=8, bs=16, dtype=torch.float32)
    args = (case.q.numpy(), case.cu_q_lens.numpy(), case.k_cache.numpy(), case.v_cache.numpy(),
            case.block_table.numpy(), case.seq_lens.numpy(), case.scale)
    out, lse = oracle.paged_prefill(*args)
    rows = [(0, 0), (19, 3), (20, 1), (28, 2), (29, 0)]
    o, l = oracle.paged_prefill_rows(*args, rows)
    for n, (t, h) in enumerate(rows):
        np.testing.assert_allclose(o[n], out[t, h], rtol=0, atol=1e-14)
        assert abs(l[n] - lse[t, h]) < 1e-14


# ---------------------------------------------------------------------------
# split-KV + log-sum-exp merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("part", [1, 16, 512, 10_000])
def test_split_then_merge_equals_unsplit(part):
    case = wl.make_decode_case(17, [1, 15, 16, 17, 600, 1100], H=4, G=2, D=16, bs=16, dtype=torch.float32)
    args = (case.q.numpy(), case.k_cache.numpy(), case.v_cache.numpy(), case.block_table.numpy(),
            case.seq_lens.numpy(), case.scale)
    o1, l1 = oracle.paged_decode(*args)
    o2, l2 = oracle.paged_decode_split(*args, part)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def test_merge_closed_forms():
    o = np.array([[[1.0, 2.0]], [[3.0, 6.0]]])               # [P=2, n=1, D=2]
    # equal lse: plain average, lse + ln 2
    out, lse = oracle.merge_states(o, np.array([[0.5], [0.5]]))
    np.testing.assert_allclose(out[0], [2.0, 4.0], rtol=0, atol=1e-15)
    assert abs(lse[0] - (0.5 + math.log(2.0))) < 1e-15
    # an empty partition weighs nothing, whatever its (never written) output holds
    o_nan = o.copy()
    o_nan[0] = np.nan
    out, lse = oracle.merge_states(o_nan, np.array([[-np.inf], [1.25]]))
    np.testing.assert_allclose(out[0], [3.0, 6.0], rtol=0, atol=0)
    assert lse[0] == 1.25
    # all empty: zero output, -inf lse
    out, lse = oracle.merge_states(o, np.array([[-np.inf], [-np.inf]]))
    assert np.array_equal(out[0], [0.0, 0.0]) and lse[0] == -np.inf
    # lse differs by ln 3: weights 1/4 and 3/4
    out, lse = oracle.merge_states(o, np.array([[0.0], [math.log(3.0)]]))
    np.testing.assert_allclose(out[0], [0.25 * 1 + 0.75 * 3, 0.25 * 2 + 0.75 * 6], rtol=0, atol=1e-15)
    assert abs(lse[0] - math.log(4.0)) < 1e-15


# ---------------------------------------------------------------------------
# MLA
# ---------------------------------------------------------------------------

def test_mla_equals_sdpa_with_value_prefix():
    rng = np.random.default_rng(51)
    H, dl, dr, bs = 8, 32, 8, 16
    lens = [1, 20, 50]
    rows = [rng.standard_normal((L, dl + dr)) for L in lens]
    pool, table = scatter_into_pages(rows, bs, rng)
    q = rng.standard_normal((len(lens), H, dl + dr))
    scale = 1.0 / math.sqrt(12.0)
    out, lse = oracle.mla_decode(q, pool, table, np.array(lens), scale, d_latent=dl)
    for s, L in enumerate(lens):
        k = np.repeat(rows[s][None], H, 0)
        v = np.repeat(rows[s][None, :, :dl], H, 0)
        ref = sdpa_f64(q[s][:, None, :].copy(), k.copy(), v.copy(), scale, causal=False)[:, 0]
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)
        for h in range(H):
            assert abs(lse[s, h] - logsumexp(scale * rows[s] @ q[s, h])) < 1e-12


def test_mla_matches_python_brute_force_small():
    rng = np.random.default_rng(53)
    H, dl, dr, bs = 3, 6, 2, 4
    lens = [3, 9]
    rows = [rng.standard_normal((L, dl + dr)) for L in lens]
    pool, table = scatter_into_pages(rows, bs, rng)
    q = rng.standard_normal((2, H, dl + dr))
    out, lse = oracle.mla_decode(q, pool, table, np.array(lens), 0.7, d_latent=dl)
    for s in range(2):
        for h in range(H):
            o, l = brute_attention(q[s, h], rows[s], rows[s][:, :dl], 0.7)
            np.testing.assert_allclose(out[s, h], o, rtol=0, atol=1e-12)
            assert abs(lse[s, h] - l) < 1e-12
