"""The give-up path of the library's bounded device waits, run on purpose.

Every pipeline wait (an mbarrier phase that a producer or the tensor cores
complete) is bounded: past its time limit it sets METIS_STATUS_WAIT_TIMEOUT in
the device status word and the kernel returns.  metis_debug_wait_probe makes
one such wait run out (its barrier expects an arrival that never comes) with a
short limit; the status bit must be set, and the context must stay usable: a
decode right after it still matches the oracle.
"""

import time

import pytest
import torch

import oracle
import paged_attention_kv_decode_gb300 as pa
from paged_attention_kv_decode_gb300 import workloads as wl
from helpers import assert_parity

pytestmark = pytest.mark.gpu

STATUS_WAIT_TIMEOUT = 4


def test_a_wait_that_nothing_completes_gives_up_and_reports():
    pa.metis_read_status(clear=True)
    t0 = time.perf_counter()
    pa.metis_debug_wait_probe(2_000_000)   # 2 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert pa.metis_read_status(clear=True) & STATUS_WAIT_TIMEOUT
    assert elapsed < 5.0                    # it gave up; it did not spin for the library's 2 s default
    # the context is still usable
    case = wl.make_decode_case(41, [1, 100, 700], H=32, G=8, D=128, bs=16, dtype=torch.bfloat16, poison=True,
                               extra_blocks=2)
    out, _ = pa.metis_paged_attn_decode(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(),
                                        case.block_table.cuda(), case.seq_lens.cuda(), case.scale,
                                        max_seq_len=case.max_seq_len)
    torch.cuda.synchronize()
    ref, _ = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, case.scale)
    assert_parity(out, ref, torch.bfloat16)
    assert pa.metis_read_status(clear=True) == 0
