"""The entry points inside CUDA graphs: captured once, replayed with new inputs.

Nothing the calls do on the host touches device memory or synchronises (TMA
descriptors are encoded on the host, shared-memory limits are raised on the
first call, the work lists are built on the device), so one warm call before
capture is all a graph needs.  Each replay gets fresh queries, lengths and
tables copied into the captured buffers and is checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_attention_kv_decode_gb300 as pa
from paged_attention_kv_decode_gb300 import workloads as wl
from helpers import assert_parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def test_split_decode_graph_replay():
    cap, P = 2048, 512
    cases = [wl.config2_batched_decode(num_seqs=12, len_lo=100 + 300 * i, len_hi=cap, extra_blocks=4)
             for i in range(3)]
    c0 = cases[0]
    S, H, D = c0.S, c0.H, c0.D
    max_blocks = cap // c0.bs
    # one cache pool big enough for every replay's tables
    nb = max(c.num_blocks for c in cases)
    kc = torch.zeros((nb, c0.bs, c0.G, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    q = torch.zeros((S, H, D), dtype=torch.bfloat16, device=DEV)
    bt = torch.full((S, max_blocks), -1, dtype=torch.int32, device=DEV)
    sl = torch.ones(S, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.metis_decode_workspace_bytes(S, H, D, cap, P), dtype=torch.uint8, device=DEV)
    call = lambda: pa.metis_paged_attn_decode(q, kc, vc, bt, sl, c0.scale, out=out, partition_size=P,
                                              max_seq_len=cap, workspace=ws)
    def load(c):
        kc[: c.num_blocks].copy_(c.k_cache)
        vc[: c.num_blocks].copy_(c.v_cache)
        q.copy_(c.q)
        bt.fill_(-1)
        bt[:, : c.block_table.shape[1]].copy_(c.block_table)
        sl.copy_(c.seq_lens)

    load(c0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                                    # warm call: raises the shared-memory limits once
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    pa.metis_read_status(clear=True)
    for c in cases:
        load(c)
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.paged_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale)
        assert_parity(out, ref, torch.bfloat16)
    assert pa.metis_read_status() == 0


def test_forward_step_graph_write_then_decode():
    """One decode step of a layer as one graph: write each sequence's new K/V row
    into its page, then attend over the cache including it."""
    c = wl.config2_batched_decode(num_seqs=8, len_lo=200, len_hi=1500)
    S, G, D, bs = c.S, c.G, c.D, c.bs
    L = c.seq_lens.numpy().astype(np.int64)
    t = L - 1
    slots = torch.from_numpy(c.block_table.numpy()[np.arange(S), t // bs].astype(np.int64) * bs + t % bs)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    q, bt, sl = c.q.to(DEV), c.block_table.to(DEV), c.seq_lens.to(DEV)
    key = torch.zeros((S, G, D), dtype=torch.bfloat16, device=DEV)
    value = torch.zeros_like(key)
    sm = slots.to(DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.metis_decode_workspace_bytes(S, c.H, D, 2048, 256), dtype=torch.uint8, device=DEV)

    def step():
        pa.metis_reshape_and_cache(key, value, kc, vc, sm)
        pa.metis_paged_attn_decode(q, kc, vc, bt, sl, c.scale, out=out, partition_size=256, max_seq_len=2048,
                                   workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator().manual_seed(21)
    ref_k, ref_v = c.k_cache, c.v_cache
    for _ in range(2):
        k_new = torch.randn(S, G, D, generator=gen).to(torch.bfloat16)
        v_new = torch.randn(S, G, D, generator=gen).to(torch.bfloat16)
        key.copy_(k_new)
        value.copy_(v_new)
        g.replay()
        torch.cuda.synchronize()
        ref_k, ref_v = oracle.reshape_and_cache(k_new, v_new, ref_k, ref_v, slots)
        ref, _ = oracle.paged_decode(c.q, ref_k, ref_v, c.block_table, c.seq_lens, c.scale)
        assert_parity(out, ref, torch.bfloat16)


def test_chunked_prefill_graph_replay():
    c = wl.make_prefill_case(77, [0, 300, 1000, 40], [200, 64, 129, 1], H=32, G=8, D=128, bs=16,
                             dtype=torch.bfloat16)
    t = [x.to(DEV) for x in (c.q, c.cu_q_lens, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
    out = torch.empty_like(t[0])
    ws = torch.empty(pa.metis_prefill_workspace_bytes(c.S, c.T, c.H, c.G), dtype=torch.uint8, device=DEV)
    call = lambda: pa.metis_paged_attn_prefill_chunk(*t, c.scale, out=out, max_seq_len=c.max_seq_len, workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    gen = torch.Generator().manual_seed(5)
    for _ in range(2):
        qn = torch.randn(c.q.shape, generator=gen).to(torch.bfloat16)
        t[0].copy_(qn)
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.paged_prefill(qn, c.cu_q_lens, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale)
        assert_parity(out, ref, torch.bfloat16)


def test_mla_graph_replay():
    c = wl.config5_mla_decode(num_seqs=6, median=300, cap=3000, extra_blocks=2)
    t = [x.to(DEV) for x in (c.q, c.kv_cache, c.block_table, c.seq_lens)]
    out = torch.empty((c.S, c.H, 512), dtype=torch.bfloat16, device=DEV)
    P = 512
    ws = torch.empty(pa.metis_mla_workspace_bytes(c.S, c.H, c.max_seq_len, P), dtype=torch.uint8, device=DEV)
    call = lambda: pa.metis_mla_decode(*t, c.scale, out=out, partition_size=P, max_seq_len=c.max_seq_len,
                                       workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    gen = torch.Generator().manual_seed(6)
    for _ in range(2):
        qn = torch.randn(c.q.shape, generator=gen).to(torch.bfloat16)
        t[0].copy_(qn)
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.mla_decode(qn, c.kv_cache, c.block_table, c.seq_lens, c.scale)
        assert_parity(out, ref, torch.bfloat16)
