"""The one-step-ahead decode pipeline: every step's output, copied back to the
host while later steps run, equals the oracle on that step's inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_attention_kv_decode_gb300 as pa
from paged_attention_kv_decode_gb300 import workloads as wl
from helpers import assert_parity

pytestmark = pytest.mark.gpu


def steps_of(case, n, seed):
    """n decode steps over one cache: new queries each step, lengths growing by one
    token a step (the new token's K/V already in the pages), shuffled block-table rows
    kept as they are."""
    g = torch.Generator().manual_seed(seed)
    S, H, D = case.q.shape
    base = case.seq_lens.clone()
    out = []
    for k in range(n):
        q = torch.randn(S, H, D, generator=g).to(case.q.dtype)
        lens = torch.clamp(base - (n - 1 - k), min=0).to(torch.int32)
        out.append((q, case.block_table.clone(), lens))
    return out


@pytest.mark.parametrize("depth,use_graph,partition", [(2, True, 0), (2, False, 0), (1, True, 0), (3, True, 0),
                                                       (2, True, 128), (2, False, 64)])
def test_every_step_matches_the_oracle(depth, use_graph, partition):
    """Depths 1-3, graphs on and off, unsplit and split-KV (decode + merge in each slot's graph)."""
    case = wl.config2_batched_decode(poison=True, num_seqs=6, len_lo=1, len_hi=600, extra_blocks=2)
    dev = torch.device("cuda")
    S, H, D = case.q.shape
    pipe = pa.DecodePipeline(case.k_cache.to(dev), case.v_cache.to(dev), S, H, case.block_table.shape[1],
                             case.scale, case.max_seq_len, partition_size=partition, depth=depth,
                             use_graph=use_graph)
    steps = steps_of(case, 7, 11 + depth)
    host_in = [(q.pin_memory(), bt.pin_memory(), sl.pin_memory()) for q, bt, sl in steps]
    host_out = [torch.empty(S, H, D, dtype=case.q.dtype).pin_memory() for _ in steps]
    events = [pipe.submit(*host_in[k], host_out[k]) for k in range(len(steps))]
    for e in events:
        e.synchronize()
    for (q, bt, sl), h in zip(steps, host_out):
        ref, _ = oracle.paged_decode(q, case.k_cache, case.v_cache, bt, sl, case.scale)
        assert_parity(h, ref, case.q.dtype)
    assert pa.metis_read_status() == 0


def test_pipeline_output_is_the_eager_output_bitwise():
    case = wl.config2_batched_decode(num_seqs=8, len_lo=100, len_hi=900)
    dev = torch.device("cuda")
    S, H, D = case.q.shape
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    pipe = pa.DecodePipeline(kc, vc, S, H, case.block_table.shape[1], case.scale, case.max_seq_len)
    h_out = torch.empty(S, H, D, dtype=case.q.dtype).pin_memory()
    pipe.submit(case.q.pin_memory(), case.block_table.pin_memory(), case.seq_lens.pin_memory(), h_out).synchronize()
    eager, _ = pa.metis_paged_attn_decode(case.q.to(dev), kc, vc, case.block_table.to(dev), case.seq_lens.to(dev),
                                          case.scale, max_seq_len=case.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(h_out, eager.cpu())


def test_layers_pick_their_own_cache():
    """Two layers' caches: step k over layer k % 2 matches the oracle on that layer."""
    case = wl.config2_batched_decode(poison=True, num_seqs=5, len_lo=1, len_hi=400, extra_blocks=2)
    g = torch.Generator().manual_seed(9)
    k2 = torch.randn(case.k_cache.shape, generator=g).to(case.k_cache.dtype)
    v2 = torch.randn(case.v_cache.shape, generator=g).to(case.v_cache.dtype)
    dev = torch.device("cuda")
    S, H, D = case.q.shape
    pipe = pa.DecodePipeline([case.k_cache.to(dev), k2.to(dev)], [case.v_cache.to(dev), v2.to(dev)], S, H,
                             case.block_table.shape[1], case.scale, case.max_seq_len)
    h_in = (case.q.pin_memory(), case.block_table.pin_memory(), case.seq_lens.pin_memory())
    outs = [torch.empty(S, H, D, dtype=case.q.dtype).pin_memory() for _ in range(4)]
    for k in range(4):
        pipe.submit(*h_in, outs[k], layer=k % 2)
    pipe.synchronize()
    for k in range(4):
        kc, vc = (case.k_cache, case.v_cache) if k % 2 == 0 else (k2, v2)
        ref, _ = oracle.paged_decode(case.q, kc, vc, case.block_table, case.seq_lens, case.scale)
        assert_parity(outs[k], ref, case.q.dtype)
