"""Pins of the prefix-cache oracle (no GPU).

mix64 is pinned to splitmix64's published output sequence; the chained keys to
their defining properties (equal prefixes share keys, a change in page k
changes keys k.. only, keys are independent of how the batch is split into
sequences); the lookup to a hand-worked sequence of hits and allocations.
"""
import os

import numpy as np

import oracle
from oracle.prefix_cache import SEED, MASK


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "splitmix64_seed0.txt")


def test_mix64_is_splitmix64():
    # splitmix64 seeded with 0: state += SEED, output mix64(state); the expected
    # outputs are the published ones (tests/golden/splitmix64_seed0.txt, with its source)
    want = [int(ln, 16) for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(want) == 2
    s, out = 0, []
    for _ in range(len(want)):
        s = (s + SEED) & MASK
        out.append(oracle.mix64(s))
    assert out == want


def test_equal_prefixes_share_keys_and_a_change_propagates_forward():
    rng = np.random.default_rng(0)
    bs = 16
    a = rng.integers(0, 50000, size=5 * bs + 7)
    b = a.copy()
    b[2 * bs + 3] += 1                      # a token of page 2
    ka = oracle.block_hashes(np.concatenate([a, b]), [0, len(a), 2 * len(a)], bs)
    n = 5                                   # full pages per sequence
    assert ka[:2] == ka[n:n + 2]            # pages 0, 1 equal
    assert all(ka[i] != ka[n + i] for i in range(2, n))
    assert len(set(ka[:n])) == n


def test_keys_depend_only_on_the_sequence():
    rng = np.random.default_rng(1)
    seqs = [rng.integers(0, 1000, size=n) for n in (40, 16, 3, 33)]
    bs = 8
    cu = np.cumsum([0] + [len(x) for x in seqs])
    together = oracle.block_hashes(np.concatenate(seqs), cu, bs)
    alone = sum((oracle.block_hashes(x, [0, len(x)], bs) for x in seqs), [])
    assert together == alone
    assert len(together) == sum(len(x) // bs for x in seqs)


def test_single_page_key_by_hand():
    toks = [3, 1, 4, 1]
    local = SEED
    for t in toks:
        local = oracle.mix64(local ^ t)
    assert oracle.block_hashes(toks, [0, 4], 4) == [oracle.mix64(0 ^ local)]


def test_lookup_hand_worked():
    table = {111: 7}
    free = [0, 1, 2]                        # top of the stack is the last element
    ref = np.zeros(10, dtype=np.int64)
    ref[7] = 2
    pages, hits, t2, f2, r2 = oracle.lookup_or_allocate([111, 222, 222, 333, 444, 111], table, free, ref)
    assert pages == [7, 2, 2, 1, 0, 7]
    assert hits == [True, False, True, False, False, True]
    assert t2 == {111: 7, 222: 2, 333: 1, 444: 0} and f2 == []
    assert list(r2[[0, 1, 2, 7]]) == [1, 1, 2, 4]
    assert table == {111: 7} and free == [0, 1, 2] and ref[7] == 2   # inputs untouched


def test_lookup_with_empty_free_stack():
    pages, hits, t2, f2, _ = oracle.lookup_or_allocate([5, 6, 5], {}, [9], np.zeros(10, dtype=np.int64))
    assert pages == [9, -1, 9] and hits == [False, False, True] and t2 == {5: 9}
