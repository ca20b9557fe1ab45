"""GPU parity of the paged KV-cache write against the oracle: a byte copy, so
every comparison is bitwise (the caches start as NaN so that a row written to
the wrong place, or not written, shows)."""
import numpy as np
import pytest
import torch

import oracle
import paged_attention_kv_decode_gb300 as pa
from paged_attention_kv_decode_gb300 import workloads as wl
from helpers import assert_parity

DEV = torch.device("cuda")

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def make(N, G, D, bs, nb, dtype, pad_frac, seed):
    g = torch.Generator().manual_seed(seed)
    key = torch.randn(N, G, D, generator=g).to(dtype)
    value = torch.randn(N, G, D, generator=g).to(dtype)
    slots = torch.randperm(nb * bs, generator=g)[:N].to(torch.int64)
    pad = torch.rand(N, generator=g) < pad_frac
    slots[pad] = -1
    kc = torch.full((nb, bs, G, D), float("nan")).to(dtype)
    return key, value, kc, kc.clone(), slots


@pytest.mark.parametrize("N,G,D,bs,dtype", [
    (3000, 8, 128, 16, torch.bfloat16),    # c2 / c4 shapes, many CTAs
    (130, 1, 64, 16, torch.float32),       # c1 shapes
    (777, 4, 64, 32, torch.bfloat16),
    (500, 2, 128, 64, torch.float32),
    (1, 8, 128, 16, torch.bfloat16),
])
def test_write_parity_bitwise(N, G, D, bs, dtype):
    nb = N // bs + 7
    key, value, kc, vc, slots = make(N, G, D, bs, nb, dtype, 0.1, N)
    ref_k, ref_v = oracle.reshape_and_cache(key, value, kc, vc, slots)
    gk, gv = kc.to(DEV), vc.to(DEV)
    pa.metis_reshape_and_cache(key.to(DEV), value.to(DEV), gk, gv, slots.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(bits(gk.cpu()), bits(ref_k))
    assert torch.equal(bits(gv.cpu()), bits(ref_v))
    assert pa.metis_read_status() == 0


def test_empty_write_changes_nothing():
    key, value, kc, vc, slots = make(4, 8, 128, 16, 3, torch.bfloat16, 0.0, 1)
    gk = kc.to(DEV)
    pa.metis_reshape_and_cache(key[:0].to(DEV), value[:0].to(DEV), gk, vc.to(DEV), slots[:0].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(bits(gk.cpu()), bits(kc))


def test_slot_past_the_pool_is_flagged_and_not_written():
    key, value, kc, vc, slots = make(40, 8, 128, 16, 5, torch.bfloat16, 0.0, 2)
    bad = slots.clone()
    bad[7] = 5 * 16 + 3                          # one past the pool
    gk, gv = kc.to(DEV), vc.to(DEV)
    pa.metis_read_status(clear=True)
    pa.metis_reshape_and_cache(key.to(DEV), value.to(DEV), gk, gv, bad.to(DEV))
    assert pa.metis_read_status() & pa.STATUS_BAD_BLOCK_ID
    keep = bad.clone()
    keep[7] = -1
    ref_k, _ = oracle.reshape_and_cache(key, value, kc, vc, keep)
    assert torch.equal(bits(gk.cpu()), bits(ref_k))


def test_write_then_decode():
    """One decode step: write each sequence's newest token with the kernel, then
    attend; equals the oracle decode over the oracle-written cache."""
    case = wl.config2_batched_decode(num_seqs=8, len_lo=100, len_hi=900)
    S, G, D, bs = case.S, case.G, case.D, case.bs
    L = case.seq_lens.numpy().astype(np.int64)
    bt = case.block_table.numpy()
    t = L - 1
    slots = torch.from_numpy(bt[np.arange(S), t // bs].astype(np.int64) * bs + t % bs)
    g = torch.Generator().manual_seed(9)
    key = torch.randn(S, G, D, generator=g).to(torch.bfloat16)
    value = torch.randn(S, G, D, generator=g).to(torch.bfloat16)
    ref_k, ref_v = oracle.reshape_and_cache(key, value, case.k_cache, case.v_cache, slots)
    ref_o, _ = oracle.paged_decode(case.q, ref_k, ref_v, case.block_table, case.seq_lens, case.scale)
    gk, gv = case.k_cache.to(DEV), case.v_cache.to(DEV)
    pa.metis_reshape_and_cache(key.to(DEV), value.to(DEV), gk, gv, slots.to(DEV))
    out, _ = pa.metis_paged_attn_decode(case.q.to(DEV), gk, gv, case.block_table.to(DEV), case.seq_lens.to(DEV),
                                        case.scale)
    torch.cuda.synchronize()
    assert_parity(out, ref_o, torch.bfloat16)


def test_mla_write_parity_bitwise():
    g = torch.Generator().manual_seed(5)
    N, bs, nb = 1000, 64, 20
    kv_c = torch.randn(N, 512, generator=g).to(torch.bfloat16)
    k_pe = torch.randn(N, 64, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:N].to(torch.int64)
    slots[::9] = -1
    cache = torch.full((nb, bs, 576), float("nan")).to(torch.bfloat16)
    ref = oracle.mla_reshape_and_cache(kv_c, k_pe, cache, slots)
    gc = cache.to(DEV)
    pa.metis_mla_reshape_and_cache(kv_c.to(DEV), k_pe.to(DEV), gc, slots.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(bits(gc.cpu()), bits(ref))


def test_full_step_write_chunked_prefill_rows():
    """The measured workload: the 8240 new rows of the chunked-prefill step (16
    chunks of 512 + 48 decodes), written where the block tables put them."""
    case = wl.config4_chunked_prefill()
    cu = case.cu_q_lens.numpy()
    L = case.seq_lens.numpy().astype(np.int64)
    bt = case.block_table.numpy()
    slots = []
    for s in range(case.S):
        ql = int(cu[s + 1] - cu[s])
        t = np.arange(L[s] - ql, L[s])
        slots.append(bt[s, t // case.bs].astype(np.int64) * case.bs + t % case.bs)
    slots = torch.from_numpy(np.concatenate(slots))
    g = torch.Generator().manual_seed(12)
    key = torch.randn(case.T, case.G, case.D, generator=g).to(torch.bfloat16)
    value = torch.randn(case.T, case.G, case.D, generator=g).to(torch.bfloat16)
    ref_k, ref_v = oracle.reshape_and_cache(key, value, case.k_cache, case.v_cache, slots)
    gk, gv = case.k_cache.to(DEV), case.v_cache.to(DEV)
    pa.metis_reshape_and_cache(key.to(DEV), value.to(DEV), gk, gv, slots.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(bits(gk.cpu()), bits(ref_k))
    assert torch.equal(bits(gv.cpu()), bits(ref_v))
