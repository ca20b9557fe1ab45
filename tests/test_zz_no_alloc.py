"""The decode entry point that allocates nothing (metis_paged_attn_decode_noalloc).

Some callers cannot call cudaMalloc: a host framework that owns all device
memory and gives its plugins no allocator, or a latency-critical path that
cannot take an allocation's implicit synchronisation.  For them the library
keeps its split-KV scratch in a static device array of
METIS_NOALLOC_SCRATCH_BYTES.  Each case is checked against the float64 CPU
oracle at the parity tolerances, and against metis_paged_attn_decode (the
same call with a caller-owned workspace).  This file is collected last so
that a run that stops at the first failure has already run every other test.
"""

import ctypes

import pytest
import torch

import oracle
import paged_attention_kv_decode_gb300 as pa
from paged_attention_kv_decode_gb300 import workloads as wl
from helpers import BF16_ATOL, BF16_RTOL, F32_ATOL, assert_lse, assert_parity


def _on_gpu(case):
    return (case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), case.block_table.cuda(), case.seq_lens.cuda())


def _run_in_a_row(cases):
    """Every case through the no-allocation call, back to back on one stream, then checked."""
    dev_in = [_on_gpu(c) for c, _ in cases]
    outs = []
    for (case, P), (q, kc, vc, bt, sl) in zip(cases, dev_in):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        pa.metis_paged_attn_decode_noalloc(q, kc, vc, bt, sl, case.scale, out=out, lse_out=lse,
                                           partition_size=P, max_seq_len=case.max_seq_len)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert pa.metis_read_status(clear=True) == 0
    for (case, P), (q, kc, vc, bt, sl), (out, lse) in zip(cases, dev_in, outs):
        ref, ref_lse = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                                           case.scale)
        assert_parity(out, ref, case.dtype)
        assert_lse(lse, ref_lse, case.dtype)
        # and within the same tolerance of the entry point that takes a caller-owned workspace
        other, other_lse = pa.metis_paged_attn_decode(q, kc, vc, bt, sl, case.scale, partition_size=P,
                                                      max_seq_len=case.max_seq_len, want_lse=True)
        torch.cuda.synchronize()
        a, b = out.double(), other.double()
        if case.dtype == torch.float32:
            assert (a - b).abs().max() <= F32_ATOL
        else:
            assert ((a - b).abs() <= BF16_ATOL + BF16_RTOL * b.abs()).all(), (a - b).abs().max()
        assert ((lse - other_lse).abs() <= 1e-3).all()


@pytest.mark.gpu
def test_noalloc_bf16_split_two_calls_in_a_row():
    # two different batches and split sizes, back to back: the second call must
    # not depend on what the first left in the shared scratch
    _run_in_a_row([(wl.config2_batched_decode(num_seqs=12, len_lo=17, len_hi=3000, poison=True, extra_blocks=5), 512),
                   (wl.make_decode_case(21, [1, 16, 17, 700, 2049, 5000], H=32, G=8, D=128, bs=16,
                                        dtype=torch.bfloat16, poison=True, extra_blocks=3), 128)])


@pytest.mark.gpu
def test_noalloc_fp32_split_then_unsplit_bf16():
    # the fp32 path (1e-5) split into 16-token partitions, then an unsplit bf16
    # call (partition_size 0: no scratch at all) right after it
    _run_in_a_row([(wl.make_decode_case(23, [1, 5, 16, 33, 64, 97], H=4, G=1, D=64, bs=16, dtype=torch.float32,
                                        poison=True, extra_blocks=2), 16),
                   (wl.config2_batched_decode(num_seqs=8, len_lo=1, len_hi=2100, poison=True, extra_blocks=2), 0)])


def test_noalloc_rejects_a_split_larger_than_the_static_scratch():
    lib = pa.load_library()
    fake = ctypes.c_void_p(0x7F0000000000)   # never dereferenced: the call is rejected first
    # 64 seqs x 32 heads x ceil(1e6 / 16) partitions x 128 floats is far beyond 64 MiB
    rc = lib.metis_paged_attn_decode_noalloc(fake, fake, fake, fake, fake, fake, None, 64, 32, 8, 128, 16, 65536,
                                             70000, pa.METIS_BF16, 0.088, 16, 1_000_000, None)
    assert rc == -5
    assert "static scratch" in pa.metis_last_error()
