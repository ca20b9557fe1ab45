#!/usr/bin/env python3
"""Throughput of paged-attention decode on one GB300 (one JSON line on stdout).

Workload: batched paged decode in bf16 -- 64 sequences with lengths drawn
U[512, 4096], 32 query heads over 8 KV heads, head_dim 128, 16-token pages
placed by a random permutation of the block pool (seeded, synthetic).  One
step is one pass of the whole decode path over the batch: one decode call
(block-table walk, paged K/V gather, QK^T, online softmax, PV, finalise),
unsplit with the longest sequences first (``--partition P`` > 0 times the
split-KV partial kernel and the log-sum-exp merge instead).  The KV cache
(604 MB) is larger than L2, and
L2 is additionally flushed between timed steps, outside the timed events, by
reading a 2x-L2 buffer (``--flush write`` zeroes it instead; that leaves L2
full of dirty lines whose write-back lands inside the next timed step, ~8 %
slower; the line reports that variant under ``flush_reference``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The line also carries ``workloads``: the tiny fp32 decode, the long-context
split-KV decode (GB/s), the chunked prefill mixed with decodes (TFLOP/s against
the measured bf16 peak), the MLA decode (TFLOP/s and GB/s), the paged KV
write of the chunked-prefill step's new rows (GB/s) and the prefix-cache page
keys + lookup over 4096 prompts sharing system prompts (tokens/s), each timed
the same way as one call of its entry point.

``value`` is decode KV GB/s: the algorithmic bytes of a step (every cached
token's K and V row for its KV head, the queries, outputs, block-table
entries and lengths; partials are overhead and not counted) divided by the
step's device time.  ``--impl reference`` times the float64 CPU oracle on a
bounded sample of the same workload instead.
"""

import os

# The oracle legs spread sequences over a pool of threads, one per host core
# (NumPy and torch release the GIL in the gathers and products); each product
# is small (4 rows x a few thousand keys), and a multi-threaded BLAS on such
# products measured ~10x slower than one thread, so BLAS runs single-threaded
# inside each worker (set before numpy loads BLAS).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% of HBM peak) and tokens/s; prefill TFLOP/s, 1 GB300"
WORKLOAD = ("batched paged decode, bf16 KV: 64 seqs, seq_lens U[512,4096], 32 q / 8 kv heads, head_dim 128, "
            "block_size 16, block_table a random permutation of the pool")
PARTITION = 0      # unsplit: one CTA per (sequence, kv head), longest sequences first (no merge)
MLA_PARTITION = 2048
E2E_LAYERS = 4      # distinct layer caches the pipelined end-to-end leg cycles through
NOMINAL_HBM_GBS = 8000.0   # nominal GB300 HBM3e bandwidth; fractions are reported against it and the measured peak
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TC_TFLOPS = (1900.0, 1700.0)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def decode_algorithmic_bytes(case) -> int:
    """K and V rows of every cached token (per KV head) + q + out + block-table entries + lengths."""
    esize = case.k_cache.element_size()
    lens = case.seq_lens.numpy().astype(np.int64)
    kv = int(lens.sum()) * case.G * case.D * 2 * esize
    qo = 2 * case.S * case.H * case.D * case.q.element_size()
    table = int(sum(-(-int(L) // case.bs) for L in lens)) * 4 + 4 * case.S
    return kv + qo + table


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_tc_peaks():
    """bf16 dense TFLOP/s: (burst, sustained)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"])), "measured"
    except Exception:
        return FALLBACK_TC_TFLOPS, "fallback"


def source_hash() -> str:
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh"):
        with open(os.path.join(ROOT, "paged_attention_kv_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "decode_bf16_kernel_batched_decode.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != source_hash():
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples (100 ms) while the GPU works."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append((time.time(), parts))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        rows = [p for _, p in self.rows if not self.uuid or self.uuid in p[1]] or [p for _, p in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable: no nvidia-smi samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in rows if num(p[2]) is not None]
        smax = [num(p[3]) for p in rows if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in rows for i in range(4) if p[6 + i].lower() == "active"})
        busy = [x for x in sm if smax and x > 0.5 * max(smax)] or sm
        return {"sm_mhz": float(np.median(busy)) if busy else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(p[4]) or 0.0) for p in rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def oracle_step(case, seqs, pool=None):
    """The oracle, as it stands, over the listed sequences: one call per sequence, spread over `pool`.
    Returns the per-sequence ``(out [1, H, D], lse [1, H])`` in the order of `seqs`."""
    import oracle

    def one(s):
        sl = slice(int(s), int(s) + 1)
        return oracle.paged_decode(case.q[sl], case.k_cache, case.v_cache, case.block_table[sl], case.seq_lens[sl],
                                   case.scale)

    if pool is None:
        return [one(s) for s in seqs]
    return list(pool.map(one, list(seqs)))


# Parity bar: fp32 max |d| <= 1e-5; bf16 inputs |d| <= 1.5e-2 + 1e-2 |ref| elementwise.
def error_summary(got: torch.Tensor, ref: np.ndarray, fp32: bool) -> dict:
    """Max abs error of a GPU output against the oracle's, and the worst error as a fraction of the bar."""
    g = got.detach().to("cpu", torch.float64).numpy()
    d = np.abs(g - ref)
    bound = np.full_like(ref, 1e-5) if fp32 else 1.5e-2 + 1e-2 * np.abs(ref)
    ratio = float((d / bound).max()) if d.size else 0.0
    return {"max_abs_err": float(d.max()) if d.size else 0.0, "tol": "1e-5 abs" if fp32 else "1.5e-2 + 1e-2 |ref|",
            "tol_ratio": ratio, "within_tol": bool(np.isfinite(g).all() and ratio <= 1.0), "outputs_checked": int(d.size)}


def sub_bytes(case, seqs) -> int:
    from paged_attention_kv_decode_gb300 import workloads as wl
    sub = wl.DecodeCase(name="sample", q=case.q[seqs], k_cache=case.k_cache, v_cache=case.v_cache,
                        block_table=case.block_table[seqs], seq_lens=case.seq_lens[seqs], scale=case.scale)
    return decode_algorithmic_bytes(sub)


def _timed_passes(case, seqs, budget_s, pool):
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(case, seqs, pool)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return reps, time.perf_counter() - t0


def cpu_baseline(case, budget_s=10.0, gpu_out=None):
    """The oracle, as it stands, on the whole batch repeated until ~budget_s of wall time, its sequences
    spread over one thread per host core; the same on one thread is reported beside it.  With `gpu_out`,
    the oracle's output of the batch is also the parity reference of the GPU step's output."""
    from concurrent.futures import ThreadPoolExecutor
    torch.set_num_threads(1)
    seqs = np.arange(case.S)
    nbytes = decode_algorithmic_bytes(case)
    cores = host_cores()
    with ThreadPoolExecutor(cores) as pool:
        reps, dt = _timed_passes(case, seqs, budget_s, pool)
        parity = None
        if gpu_out is not None:
            ref = np.concatenate([o for o, _ in oracle_step(case, seqs, pool)])
            parity = error_summary(gpu_out, ref, case.dtype == torch.float32)
    reps1, dt1 = _timed_passes(case, seqs, budget_s / 2, None)
    return {"value": nbytes * reps / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "parity_of_gpu_output": parity,
            "sample": f"the full 64-sequence batch, {reps} pass(es) in {dt:.1f} s wall, one oracle call per "
                      f"sequence over {cores} threads (float64 NumPy, BLAS single-threaded per call)",
            "single_thread": {"value": nbytes * reps1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"the same batch, {reps1} pass(es) in {dt1:.1f} s on one thread"}}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor
    from paged_attention_kv_decode_gb300 import workloads as wl
    torch.set_num_threads(1)
    case = wl.config2_batched_decode()
    cores = host_cores()
    rng = np.random.default_rng(0)
    with ThreadPoolExecutor(cores) as pool:
        t0 = time.perf_counter()
        oracle_step(case, np.arange(min(cores, case.S)), pool)
        per_seq = max((time.perf_counter() - t0) / min(cores, case.S), 1e-4)
        budget = 150.0
        n = int(max(1, min(case.S, budget / max(1, args.steps + args.warmup) / per_seq)))
        samples = [rng.choice(case.S, size=n, replace=False) for _ in range(args.steps + args.warmup)]
        for i in range(args.warmup):
            oracle_step(case, samples[i], pool)
        tot_bytes = 0
        t0 = time.perf_counter()
        for i in range(args.steps):
            s = samples[args.warmup + i]
            oracle_step(case, s, pool)
            tot_bytes += sub_bytes(case, s)
        dt = time.perf_counter() - t0
    value = tot_bytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_seqs_per_step": n},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} of 64 sequences per step (random), one oracle call per sequence over "
                                       f"{cores} threads, float64 NumPy"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

class L2Flush:
    """Evicts L2 between timed steps, outside the timed events, by touching a buffer of
    twice its size: "read" sums the buffer (L2 is left holding clean lines, as after a
    model's weight reads), "write" zeroes it (L2 is left holding dirty lines, whose
    write-back then falls inside the next timed step)."""

    def __init__(self, nbytes, dev, mode):
        self.buf = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)
        self.mode = mode

    def __call__(self):
        if self.mode == "write":
            self.buf.zero_()
        else:
            self.buf.sum(dtype=torch.int64)


def run_ours(args, world, rank, local):
    import paged_attention_kv_decode_gb300 as pa
    from paged_attention_kv_decode_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = wl.config2_batched_decode()
    P = args.partition
    S, H, D = case.S, case.H, case.D
    max_len = case.max_seq_len
    q = case.q.to(dev)
    kc = case.k_cache.to(dev)
    vc = case.v_cache.to(dev)
    bt = case.block_table.to(dev)
    sl = case.seq_lens.to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(max(256, pa.metis_decode_workspace_bytes(S, H, D, max_len, P)), dtype=torch.uint8, device=dev)
    part_out, part_lse = pa.split_workspace_views(ws, S, H, D, max_len, P) if P > 0 else (None, None)
    nbytes = decode_algorithmic_bytes(case)
    props = torch.cuda.get_device_properties(dev)
    flush = L2Flush(max(2 * int(getattr(props, "L2_cache_size", 128 << 20)), 256 << 20), dev, args.flush)
    stream = torch.cuda.current_stream(dev)

    def step():
        if P == 0:   # one launch: the decode kernel writes the output directly
            pa.metis_paged_attn_decode(q, kc, vc, bt, sl, case.scale, out=out, partition_size=0, max_seq_len=max_len,
                                       stream=stream)
            ev_mid.record(stream)
            return
        pa.metis_paged_attn_decode_partials(q, kc, vc, bt, sl, case.scale, partition_size=P, max_seq_len=max_len,
                                            workspace=ws, stream=stream)
        ev_mid.record(stream)
        pa.metis_merge_attn_states(part_out, part_lse, sl, P, out=out, stream=stream)

    ev_mid = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    # clock ramp (untimed; ~1 s, or a fixed number of steps so that profiler launch indices are fixed),
    # then W warm-up steps
    if args.ramp_steps is not None:
        for _ in range(args.ramp_steps):
            step()
        torch.cuda.synchronize()
    else:
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pa.metis_read_status(clear=True)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark()
    for i in range(args.steps):
        flush()                      # untimed: evict L2 between steps
        starts[i].record(stream)
        ev_mid = mids[i]
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sampler.mark()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kern_ms = [s.elapsed_time(m) for s, m in zip(starts, mids)]
    status = pa.metis_read_status(clear=True)
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = world * nbytes * args.steps / (total_ms * 1e-3) / 1e9
    kern_avg_ms = float(np.mean(kern_ms))
    merge_avg_ms = float(np.mean([a - b for a, b in zip(step_ms, kern_ms)]))

    # reference: the same steps with the other flush (untimed either way)
    other = "write" if flush.mode == "read" else "read"
    ref_flush = L2Flush(flush.buf.numel() * 4, dev, other)
    ref_n = min(args.steps, 50)
    r_s = [torch.cuda.Event(enable_timing=True) for _ in range(ref_n)]
    r_e = [torch.cuda.Event(enable_timing=True) for _ in range(ref_n)]
    for i in range(ref_n):
        ref_flush()
        r_s[i].record(stream)
        ev_mid = mids[i]
        step()
        r_e[i].record(stream)
    torch.cuda.synchronize()
    ref_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(r_s, r_e)), world, dev)
    del ref_flush

    # end to end through the public call: pinned host inputs -> device, decode, output -> pinned host
    h_q = case.q.pin_memory()
    h_bt = case.block_table.pin_memory()
    h_sl = case.seq_lens.pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    d_q, d_bt, d_sl = torch.empty_like(q), torch.empty_like(bt), torch.empty_like(sl)
    e2e_n = args.steps
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_n)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_n)]

    def e2e_step(i):
        e_s[i].record(stream)
        d_q.copy_(h_q, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        pa.metis_paged_attn_decode(d_q, kc, vc, d_bt, d_sl, case.scale, out=out, partition_size=P,
                                   max_seq_len=max_len, workspace=ws, stream=stream)
        h_out.copy_(out, non_blocking=True)
        e_e[i].record(stream)

    for i in range(min(3, e2e_n)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    for i in range(e2e_n):
        flush()
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)), world, dev)

    # the same steps through the one-step-ahead pipeline: step k + 1's inputs go in and
    # step k's output comes back while the decodes run.  Consecutive steps decode
    # different layers (four caches of this shape, 2.4 GB), as a model's decode step
    # would, so that nothing a step reads is still in L2 for the next and the steps
    # can run back to back without a flush.
    layers_k, layers_v = [kc], [vc]
    gen = torch.Generator(device=dev).manual_seed(77)
    for _ in range(E2E_LAYERS - 1):
        layers_k.append(torch.randn(kc.shape, generator=gen, device=dev).to(kc.dtype))
        layers_v.append(torch.randn(vc.shape, generator=gen, device=dev).to(vc.dtype))
    pipe = pa.DecodePipeline(layers_k, layers_v, S, H, bt.shape[1], case.scale, max_len, partition_size=P, depth=2)
    h_outs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    for i in range(3):
        pipe.submit(h_q, h_bt, h_sl, h_outs[i % 2], layer=i % E2E_LAYERS)
    pipe.synchronize()
    barrier(world)
    p_start = torch.cuda.Event(enable_timing=True)
    p_end = torch.cuda.Event(enable_timing=True)
    p_start.record(pipe.copy_in)
    for i in range(e2e_n):
        pipe.submit(h_q, h_bt, h_sl, h_outs[i % 2], layer=i % E2E_LAYERS)
    p_end.record(pipe.copy_out)
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    sampler.stop()
    pipe_ms = max_over_ranks(p_start.elapsed_time(p_end), world, dev)
    h2d = h_q.numel() * h_q.element_size() + h_bt.numel() * 4 + h_sl.numel() * 4
    d2h = h_out.numel() * h_out.element_size()

    if rank != 0:
        return 0
    graph_line = graph_replay(q, kc, vc, bt, sl, out, ws, case.scale, P, max_len, nbytes, args.steps, flush, world,
                              dev)
    peak, peak_src = load_peaks()
    achieved = nbytes / (kern_avg_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "partition_size": P, "tokens": int(case.seq_lens.sum()),
                   "kv_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2 (KV 604 MB) and L2 flushed between timed steps (untimed 2x-L2 "
                         f"{flush.mode}: {'clean lines, as after weight reads' if flush.mode == 'read' else 'dirty lines, written back inside the next step'})",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": world * S * args.steps / (total_ms * 1e-3),
        "flush_reference": {"flush": other, "value": world * nbytes * ref_n / (ref_ms * 1e-3) / 1e9,
                            "ms_per_step": ref_ms / ref_n, "steps": ref_n},
        "hbm_frac": value / peak,
        "hbm_frac_nominal": value / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": "decode_bf16_kernel", "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(), "kernel_ms": kern_avg_ms, "merge_ms": merge_avg_ms if P > 0 else None,
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": world * nbytes * e2e_n / (pipe_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": pipe_ms / e2e_n,
                "note": "KV cache resident in HBM; per step: q, block table, lengths H2D from pinned memory, "
                        "output D2H to pinned memory, through DecodePipeline (two slots: a step's copies "
                        "overlap the neighbouring steps' decodes, each decode a replayed CUDA graph); "
                        "consecutive steps decode four layers' caches in turn (2.4 GB, no L2 reuse), "
                        "timed from the first copy to the last read-back; unlike `value`, NO L2 flush runs "
                        "between these steps (they run back to back), so a step may start while the previous "
                        "one drains",
                "serial": {"value": world * nbytes * e2e_n / (e2e_ms * 1e-3) / 1e9, "ms_per_step": e2e_ms / e2e_n,
                           "note": "the same step with copies, decode and read-back one after another on one "
                                   "stream, L2 flushed between steps"}},
        "graph": graph_line,
        "gpu_launches": (2 if P > 0 else 1) * args.steps,
        "device_status": status,
        "clocks": sampler.summary(),
    }
    if args.workloads:
        (tcb, tcs), tc_src = load_tc_peaks()
        names = [w.strip() for w in args.workloads.split(",") if w.strip()]
        line["workloads"] = other_workloads(names, args.workload_reps, dev, flush, stream, peak, (tcb, tcs),
                                            oracle_legs=not args.no_cpu_baseline, c3_seqs=args.c3_seqs)
        line["workloads"]["peaks"] = {"hbm_GB_s": peak, "bf16_TFLOP_s_burst": tcb, "bf16_TFLOP_s_sustained": tcs,
                                      "source": tc_src}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, gpu_out=out)
        line["max_abs_err"] = line["cpu_baseline"]["parity_of_gpu_output"]["max_abs_err"]
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def graph_replay(q, kc, vc, bt, sl, out, ws, scale, P, max_len, nbytes, steps, flush, world, dev):
    """The same decode step captured once as a CUDA graph and replayed `steps` times
    (informational: launch overhead removed; with a split step, no event sits
    between the two launches, so the merge's launch overlaps the decode tail)."""
    import paged_attention_kv_decode_gb300 as pa
    try:
        call = lambda: pa.metis_paged_attn_decode(q, kc, vc, bt, sl, scale, out=out, partition_size=P,
                                                  max_seq_len=max_len, workspace=ws)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream(dev)
        ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world)
        for i in range(steps):
            flush()
            ev_s[i].record(cur)
            g.replay()
            ev_e[i].record(cur)
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_e)), world, dev)
        return {"value": world * nbytes * steps / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms / steps,
                "note": "the timed step captured as one CUDA graph and replayed"}
    except Exception as e:  # noqa: BLE001 -- reported, never fatal for the bench line
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


# the other workloads: timed the same way (events, untimed L2 flush between reps)
# ---------------------------------------------------------------------------

def _time_calls(call, reps, flush, stream, name=None):
    """Median and min event time of `call` over `reps` (3 untimed calls first, L2 flushed before each
    timed one).  With `name`, the calls sit in an NVTX range of that name, so a profiler can pick out
    this workload's launches (ncu --nvtx --nvtx-include "<name>/")."""
    if name:
        torch.cuda.nvtx.range_push(name)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    if name:
        torch.cuda.nvtx.range_pop()
    return float(np.median(ts)), float(np.min(ts))


def oracle_leg(items, fn, work, unit, fp32, gpu_out, note):
    """CPU leg of a workload: the oracle, as it stands, called once per item (a sequence, or a sub-batch of
    one sequence) over one thread per host core, timed; its output is the parity reference of `gpu_out`
    (rows in item order).  `work` is the workload's work in `unit` x 1e9 (bytes or flops)."""
    from concurrent.futures import ThreadPoolExecutor
    torch.set_num_threads(1)
    cores = host_cores()
    with ThreadPoolExecutor(cores) as pool:
        t0 = time.perf_counter()
        res = list(pool.map(fn, items))
        dt = time.perf_counter() - t0
    ref = np.concatenate(res)
    return {"value": work / dt / 1e9, "unit": unit, "cores": cores, "kind": "oracle", "wall_s": dt,
            "sample": note, "parity_of_gpu_output": error_summary(gpu_out, ref, fp32)}


def other_workloads(names, reps, dev, flush, stream, peak_hbm, peaks_tc, oracle_legs=True, c3_seqs=8):
    import paged_attention_kv_decode_gb300 as pa
    from paged_attention_kv_decode_gb300 import workloads as wl
    res = {}
    tc_burst, tc_sus = peaks_tc
    if "c1" in names:
        c = wl.config1_tiny_decode()
        t = [x.to(dev) for x in (c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
        out = torch.empty_like(t[0])
        med, mn = _time_calls(lambda: pa.metis_paged_attn_decode(*t, c.scale, out=out, max_seq_len=c.max_seq_len,
                                                                  stream=stream), reps, flush, stream,
                              "tiny_decode_fp32")
        nb = decode_algorithmic_bytes(c)
        # the same call captured as a CUDA graph: the device time without the host's issue time
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            pa.metis_paged_attn_decode(*t, c.scale, out=out, max_seq_len=c.max_seq_len)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pa.metis_paged_attn_decode(*t, c.scale, out=out, max_seq_len=c.max_seq_len)
        torch.cuda.synchronize()
        gmed, _ = _time_calls(g.replay, reps, flush, stream)
        res["tiny_decode_fp32"] = {"ms": med, "GB_s": nb / med / 1e6, "graph_ms": gmed, "kv_bytes": nb,
                                   "note": "about 67 KB of KV: launch-latency bound (ms: issued from Python; "
                                           "graph_ms: replayed as a CUDA graph)"}
        if oracle_legs:
            import oracle
            res["tiny_decode_fp32"]["cpu_baseline"] = oracle_leg(
                range(c.S), lambda si: oracle.paged_decode(c.q[si:si + 1], c.k_cache, c.v_cache,
                                                           c.block_table[si:si + 1], c.seq_lens[si:si + 1],
                                                           c.scale)[0],
                nb, "GB/s", True, out, "every sequence, one oracle call each")
    if "c3" in names:
        c = wl.config3_long_split_decode(num_seqs=c3_seqs)
        t = [x.to(dev) for x in (c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
        out = torch.empty_like(t[0])
        ws = torch.empty(pa.metis_decode_workspace_bytes(c.S, c.H, c.D, c.max_seq_len, c.partition_size),
                         dtype=torch.uint8, device=dev)
        med, mn = _time_calls(lambda: pa.metis_paged_attn_decode(*t, c.scale, out=out, partition_size=c.partition_size,
                                                                  max_seq_len=c.max_seq_len, workspace=ws,
                                                                  stream=stream), reps, flush, stream,
                              "long_split_decode")
        nb = decode_algorithmic_bytes(c)
        res["long_split_decode"] = {"ms": med, "GB_s": nb / med / 1e6, "hbm_frac": nb / med / 1e6 / peak_hbm,
                                    "hbm_frac_nominal": nb / med / 1e6 / NOMINAL_HBM_GBS,
                                    "kv_bytes": nb, "partition_size": c.partition_size,
                                    "tokens_per_s": c.S / (med * 1e-3)}
        if oracle_legs:
            import oracle
            res["long_split_decode"]["cpu_baseline"] = oracle_leg(
                range(c.S), lambda si: oracle.paged_decode(c.q[si:si + 1], c.k_cache, c.v_cache,
                                                           c.block_table[si:si + 1], c.seq_lens[si:si + 1],
                                                           c.scale)[0],
                nb, "GB/s", False, out, "every sequence (unsplit oracle), one oracle call each")
        del t, out, ws, c
        torch.cuda.empty_cache()
    if "c4" in names:
        c = wl.config4_chunked_prefill()
        t = [x.to(dev) for x in (c.q, c.cu_q_lens, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
        out = torch.empty_like(t[0])
        ws = torch.empty(pa.metis_prefill_workspace_bytes(c.S, c.T, c.H, c.G), dtype=torch.uint8, device=dev)
        med, mn = _time_calls(lambda: pa.metis_paged_attn_prefill_chunk(*t, c.scale, out=out, max_seq_len=c.max_seq_len,
                                                                        workspace=ws, stream=stream), reps, flush,
                              stream, "chunked_prefill")
        cu = c.cu_q_lens.numpy()
        lens = c.seq_lens.numpy()
        flops = 0
        for si in range(c.S):
            ql = int(cu[si + 1] - cu[si])
            flops += int(((lens[si] - ql) + np.arange(ql) + 1).sum()) * c.H * 4 * c.D
        tf = flops / med / 1e9
        qlen = np.diff(cu)
        kv_bytes = int(lens.astype(np.int64).sum()) * c.G * c.D * 2 * 2
        io_bytes = 2 * c.T * c.H * c.D * 2                       # q in, out
        flop_ms = flops / (tc_burst * 1e9)
        byte_ms = (kv_bytes + io_bytes) / (peak_hbm * 1e6)

        def sub_call(sel, name):
            # the same call over a subset of the sequences (the chunks, or the decodes)
            rows = np.concatenate([np.arange(cu[si], cu[si + 1]) for si in sel])
            sq = c.q[torch.from_numpy(rows)].contiguous().to(dev)
            scu = torch.from_numpy(np.concatenate([[0], np.cumsum(qlen[sel])]).astype(np.int32)).to(dev)
            sbt = c.block_table[torch.from_numpy(sel)].contiguous().to(dev)
            ssl = c.seq_lens[torch.from_numpy(sel)].contiguous().to(dev)
            sout = torch.empty_like(sq)
            sws = torch.empty(pa.metis_prefill_workspace_bytes(len(sel), len(rows), c.H, c.G), dtype=torch.uint8,
                              device=dev)
            sm, _ = _time_calls(lambda: pa.metis_paged_attn_prefill_chunk(sq, scu, t[2], t[3], sbt, ssl, c.scale,
                                                                          out=sout, max_seq_len=c.max_seq_len,
                                                                          workspace=sws, stream=stream),
                                reps, flush, stream, name)
            sflops = sum(int(((lens[si] - qlen[si]) + np.arange(qlen[si]) + 1).sum()) for si in sel) * c.H * 4 * c.D
            skv = int(lens[sel].astype(np.int64).sum()) * c.G * c.D * 2 * 2
            return sm, sflops, skv

        ch_ms, ch_flops, _ = sub_call(np.where(qlen > 1)[0], "chunked_prefill_chunks")
        de_ms, _, de_kv = sub_call(np.where(qlen == 1)[0], "chunked_prefill_decodes")
        res["chunked_prefill"] = {"ms": med, "TFLOP_s": tf, "tensor_frac_burst": tf / tc_burst,
                                  "tensor_frac_sustained": tf / tc_sus, "flops": flops, "tokens": c.T,
                                  "tokens_per_s": c.T / (med * 1e-3),
                                  "flop_bound_ms": flop_ms, "byte_bound_ms": byte_ms,
                                  "roofline_frac": max(flop_ms, byte_ms) / med,
                                  "chunks_alone": {"ms": ch_ms, "TFLOP_s": ch_flops / ch_ms / 1e9,
                                                   "tensor_frac_burst": ch_flops / ch_ms / 1e9 / tc_burst},
                                  "decodes_alone": {"ms": de_ms, "GB_s": de_kv / de_ms / 1e6,
                                                    "hbm_frac": de_kv / de_ms / 1e6 / peak_hbm},
                                  "note": "one call: 16 chunks of 512 over cached prefixes + 48 single-token decodes; "
                                          "roofline_frac = max(flop bound, byte bound) / call time; the two kinds "
                                          "also timed as calls of their own"}
        if oracle_legs:
            import oracle

            def one_seq(si):
                ql = int(qlen[si])
                return oracle.paged_prefill(c.q[int(cu[si]):int(cu[si + 1])],
                                            torch.tensor([0, ql], dtype=torch.int32), c.k_cache, c.v_cache,
                                            c.block_table[si:si + 1], c.seq_lens[si:si + 1], c.scale)[0]

            # the GPU output is in the same (sequence-major) row order
            res["chunked_prefill"]["cpu_baseline"] = oracle_leg(
                range(c.S), one_seq, flops, "TFLOP/s", False, out,
                "every row of every sequence, one oracle call per sequence")
            res["chunked_prefill"]["cpu_baseline"]["value"] /= 1e3   # GFLOP/s -> TFLOP/s
        del t, out, ws, c
        torch.cuda.empty_cache()
    if "kvw" in names:
        # the paged KV write in front of the chunked-prefill step: its 8240 new K/V rows
        c = wl.config4_chunked_prefill()
        cu = c.cu_q_lens.numpy()
        lens = c.seq_lens.numpy().astype(np.int64)
        bt = c.block_table.numpy()
        slots = []
        for si in range(c.S):
            ql = int(cu[si + 1] - cu[si])
            tt = np.arange(lens[si] - ql, lens[si])
            slots.append(bt[si, tt // c.bs].astype(np.int64) * c.bs + tt % c.bs)
        slots = torch.from_numpy(np.concatenate(slots)).to(dev)
        g = torch.Generator().manual_seed(12)
        key = torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)
        value = torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)
        kc, vc = c.k_cache.to(dev), c.v_cache.to(dev)
        med, mn = _time_calls(lambda: pa.metis_reshape_and_cache(key, value, kc, vc, slots, stream=stream), reps, flush,
                              stream, "kv_write")
        nb = 2 * 2 * c.T * c.G * c.D * 2 + c.T * 8    # K and V rows read and written, plus the slots
        torch.cuda.synchronize()
        blk, off = slots // c.bs, slots % c.bs
        exact = bool(torch.equal(kc[blk, off], key) and torch.equal(vc[blk, off], value))
        # A ~12 us kernel is close to the events' resolution and its launch cost: also time
        # 40 writes back to back, over 8 input sets (545 MB: more than L2, so every call
        # reads its rows from HBM), per call
        sets = [(torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev),
                 torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev),
                 slots[torch.randperm(slots.numel(), generator=g).to(dev)]) for _ in range(8)]

        def many():
            for i in range(40):
                k_, v_, s_ = sets[i % 8]
                pa.metis_reshape_and_cache(k_, v_, kc, vc, s_, stream=stream)
        for _ in range(2):
            many()
        torch.cuda.synchronize()
        per = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            many()
            e1.record(stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / 40)
        b2b = float(np.median(per))
        res["kv_write"] = {"ms": med, "GB_s": nb / med / 1e6, "hbm_frac": nb / med / 1e6 / peak_hbm,
                           "hbm_frac_nominal": nb / med / 1e6 / NOMINAL_HBM_GBS, "bytes": nb, "tokens": c.T,
                           "written_rows_bitwise_equal_to_inputs": exact,
                           "back_to_back": {"ms": b2b, "GB_s": nb / b2b / 1e6, "hbm_frac": nb / b2b / 1e6 / peak_hbm,
                                            "note": "40 calls in a row over 8 input sets larger than L2 together, "
                                                    "per call"},
                           "note": "the chunked-prefill step's new K/V rows scattered into their pages; one call "
                                   "per event pair with L2 flushed in between (ms), and back to back"}
        del key, value, kc, vc, slots, c, sets
        torch.cuda.empty_cache()
    if "kvw_step" in names:
        # the paged K/V write chained in front of attention (the write kernel lets the
        # attention call launch early; it waits for the write before reading the cache):
        # (a) the batched-decode step: each sequence's newest token written, then decode;
        # (b) the chunked-prefill step: its 8,240 new rows written, then the mixed call
        res["kv_write_then_attention"] = {}
        c = wl.config2_batched_decode()
        t = [x.to(dev) for x in (c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
        out = torch.empty_like(t[0])
        lens = c.seq_lens.numpy().astype(np.int64)
        bt = c.block_table.numpy()
        last = lens - 1
        slots = torch.from_numpy(bt[np.arange(c.S), last // c.bs].astype(np.int64) * c.bs + last % c.bs).to(dev)
        g = torch.Generator().manual_seed(13)
        key = torch.randn(c.S, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)
        value = torch.randn(c.S, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)

        def dec():
            pa.metis_paged_attn_decode(*t, c.scale, out=out, max_seq_len=c.max_seq_len, stream=stream)

        def wdec():
            pa.metis_reshape_and_cache(key, value, t[1], t[2], slots, stream=stream)
            dec()

        d_ms, _ = _time_calls(dec, reps, flush, stream, "decode_alone")
        wd_ms, _ = _time_calls(wdec, reps, flush, stream, "write_then_decode")
        res["kv_write_then_attention"]["batched_decode"] = {
            "decode_ms": d_ms, "write_then_decode_ms": wd_ms, "added_us": (wd_ms - d_ms) * 1e3, "new_rows": c.S,
            "note": "each sequence's newest K/V row written into its page, then the unsplit decode"}
        del t, out, key, value, slots, c
        c = wl.config4_chunked_prefill()
        t = [x.to(dev) for x in (c.q, c.cu_q_lens, c.k_cache, c.v_cache, c.block_table, c.seq_lens)]
        out = torch.empty_like(t[0])
        ws = torch.empty(pa.metis_prefill_workspace_bytes(c.S, c.T, c.H, c.G), dtype=torch.uint8, device=dev)
        cu = c.cu_q_lens.numpy()
        lens = c.seq_lens.numpy().astype(np.int64)
        bt = c.block_table.numpy()
        sl = []
        for si in range(c.S):
            ql = int(cu[si + 1] - cu[si])
            tt = np.arange(lens[si] - ql, lens[si])
            sl.append(bt[si, tt // c.bs].astype(np.int64) * c.bs + tt % c.bs)
        slots = torch.from_numpy(np.concatenate(sl)).to(dev)
        key = torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)
        value = torch.randn(c.T, c.G, c.D, generator=g).to(torch.bfloat16).to(dev)

        def pf():
            pa.metis_paged_attn_prefill_chunk(*t, c.scale, out=out, max_seq_len=c.max_seq_len, workspace=ws,
                                              stream=stream)

        def wpf():
            pa.metis_reshape_and_cache(key, value, t[2], t[3], slots, stream=stream)
            pf()

        def w_only():
            pa.metis_reshape_and_cache(key, value, t[2], t[3], slots, stream=stream)

        p_ms, _ = _time_calls(pf, reps, flush, stream, "prefill_alone")
        w_ms, _ = _time_calls(w_only, reps, flush, stream, "write_alone")
        wp_ms, _ = _time_calls(wpf, reps, flush, stream, "write_then_prefill")
        res["kv_write_then_attention"]["chunked_prefill"] = {
            "prefill_ms": p_ms, "write_ms": w_ms, "write_then_prefill_ms": wp_ms,
            "added_us": (wp_ms - p_ms) * 1e3, "hidden_us": (p_ms + w_ms - wp_ms) * 1e3, "new_rows": c.T,
            "note": "the step's new K/V rows written into their pages, then the mixed chunked-prefill call"}
        del t, out, ws, key, value, slots, c
        torch.cuda.empty_cache()
    if "pfx" in names:
        # prefix-cache page keys + lookup-or-allocate over a batch of prompts sharing system prompts
        c = wl.prefix_workload()
        cap = 1 << 17
        table = pa.prefix_table_alloc(cap, dev)
        tok, cut, cup = (torch.from_numpy(x).to(dev) for x in (c.tokens, c.cu_tokens, c.cu_pages))
        stack = torch.from_numpy(c.free_stack).to(dev)
        count0 = torch.tensor([c.num_pages], dtype=torch.int32, device=dev)
        count = count0.clone()
        ref = torch.zeros(c.num_pages, dtype=torch.int32, device=dev)
        keys = torch.empty(c.total_pages, dtype=torch.int64, device=dev)
        pages = torch.empty(c.total_pages, dtype=torch.int32, device=dev)
        hits = torch.empty(c.total_pages, dtype=torch.uint8, device=dev)
        ws = torch.empty(pa.metis_prefix_lookup_workspace_bytes(c.total_pages), dtype=torch.uint8, device=dev)

        def hashes():
            pa.metis_prefix_block_hashes(tok, cut, cup, c.block_size, c.total_pages, keys_out=keys)

        def lookup():
            pa.metis_prefix_table_init(*table)
            count.copy_(count0)
            pa.metis_prefix_lookup(keys, table, stack, count, ref, pages_out=pages, hits_out=hits, workspace=ws)

        def whole():
            hashes()
            lookup()

        def as_graph(fn):
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream().wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):  # the calls above launch on the current (capturing) stream
                fn()
            torch.cuda.synchronize()
            return g

        # device time of the step: each piece captured as a CUDA graph and replayed
        # (eager calls are bound by the host's issue rate at these sizes)
        med, _ = _time_calls(as_graph(whole).replay, reps, flush, stream)
        hmed, _ = _time_calls(as_graph(hashes).replay, reps, flush, stream)
        lmed, _ = _time_calls(as_graph(lookup).replay, reps, flush, stream)
        emed, _ = _time_calls(whole, reps, flush, stream)
        torch.cuda.synchronize()
        hit_rate = float(hits.float().mean().item())
        res["prefix_lookup"] = {"ms": med, "hash_ms": hmed, "lookup_ms": lmed, "eager_ms": emed,
                                "tokens": c.num_tokens, "prompts": c.num_seqs, "pages": c.total_pages,
                                "tokens_per_s": c.num_tokens / (med * 1e-3),
                                "pages_per_s": c.total_pages / (med * 1e-3), "hit_rate": hit_rate,
                                "launches": 7,
                                "note": "one step as a CUDA graph: table reset, stack depth reset, page keys of "
                                        "every full page, lookup-or-allocate in batch order; eager_ms: the same "
                                        "step issued call by call from Python"}
        del table, tok, cut, cup, stack, count0, count, ref, keys, pages, hits, ws, c
        torch.cuda.empty_cache()
    if "c5" in names:
        c = wl.config5_mla_decode()
        t = [x.to(dev) for x in (c.q, c.kv_cache, c.block_table, c.seq_lens)]
        out = torch.empty((c.S, c.H, c.d_latent), dtype=torch.bfloat16, device=dev)
        P = MLA_PARTITION
        ws = torch.empty(pa.metis_mla_workspace_bytes(c.S, c.H, c.max_seq_len, P), dtype=torch.uint8, device=dev)
        med, mn = _time_calls(lambda: pa.metis_mla_decode(*t, c.scale, out=out, partition_size=P,
                                                          max_seq_len=c.max_seq_len, workspace=ws, stream=stream),
                              reps, flush, stream, "mla_decode")
        tok = int(c.seq_lens.sum())
        flops = tok * c.H * 2 * (576 + 512)
        nb = tok * 576 * 2 + c.S * c.H * (576 + 512) * 2 + int(sum(-(-int(L) // c.bs) for L in c.seq_lens)) * 4
        tf = flops / med / 1e9
        res["mla_decode"] = {"ms": med, "TFLOP_s": tf, "tensor_frac_burst": tf / tc_burst,
                             "tensor_frac_sustained": tf / tc_sus,
                             "GB_s": nb / med / 1e6, "hbm_frac": nb / med / 1e6 / peak_hbm,
                             "hbm_frac_nominal": nb / med / 1e6 / NOMINAL_HBM_GBS, "flops": flops,
                             "bytes": nb, "tokens": tok, "partition_size": P,
                             "tokens_per_s": c.S / (med * 1e-3)}
        if oracle_legs:
            import oracle
            res["mla_decode"]["cpu_baseline"] = oracle_leg(
                range(c.S), lambda si: oracle.mla_decode(c.q[si:si + 1], c.kv_cache, c.block_table[si:si + 1],
                                                         c.seq_lens[si:si + 1], c.scale)[0],
                flops, "TFLOP/s", False, out, "every sequence, one oracle call each")
            res["mla_decode"]["cpu_baseline"]["value"] /= 1e3   # GFLOP/s -> TFLOP/s
        del t, out, ws, c
        torch.cuda.empty_cache()
    return res


def run_workloads_only(args, local):
    """Profiling aid: the --workloads list alone, timed as in the full run, printed as one JSON object."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    flush = L2Flush(max(2 * int(getattr(props, "L2_cache_size", 128 << 20)), 256 << 20), dev, args.flush)
    peak, _ = load_peaks()
    (tcb, tcs), _ = load_tc_peaks()
    names = [w.strip() for w in args.workloads.split(",") if w.strip()]
    res = other_workloads(names, args.workload_reps, dev, flush, torch.cuda.current_stream(dev), peak, (tcb, tcs),
                          oracle_legs=not args.no_cpu_baseline, c3_seqs=args.c3_seqs)
    print(json.dumps({"workloads_only": res}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition", type=int, default=PARTITION)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="c1,c3,c4,c5,kvw,kvw_step,pfx",
                    help="other workloads to time after the main one (comma list of c1,c3,c4,c5,kvw,kvw_step,pfx; "
                         "empty: none)")
    ap.add_argument("--workload-reps", type=int, default=20)
    ap.add_argument("--skip-main", action="store_true",
                    help="profiling aid: run only the --workloads list and print it (no headline step)")
    ap.add_argument("--c3-seqs", type=int, default=8,
                    help="sequences of the long split-KV workload (8; fewer gives a smaller case for profiling)")
    ap.add_argument("--flush", choices=["read", "write"], default="read",
                    help="how L2 is evicted between timed steps (outside the timed events)")
    ap.add_argument("--ramp-steps", type=int, default=None,
                    help="untimed steps before warm-up (default: about one second of steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3 (the minimum)")
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
    elif args.skip_main:
        rc = run_workloads_only(args, local)
    else:
        rc = run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
