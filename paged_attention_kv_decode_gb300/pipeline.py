"""One-step-ahead decode pipeline over the C ABI.

A serving loop hands the decode step new queries, block tables and lengths on
the host every step and reads the output back (the scheduler drives the
kernels with the block table and sequence lengths every step: vllm-metal
article, section 4; the steps are captured as CUDA graphs: vllm-metal article,
section 5).  Done one after the other, the host<->device copies of a step sit
between two decode launches.  ``DecodePipeline`` keeps ``depth`` device slots
and three streams so that the copies of step k + 1 run while step k computes
and the output of step k returns while step k + 1 computes:

    copy-in stream   H2D q, block table, lengths of step k   -> event in_done[k]
    compute stream   wait in_done[k]; decode (a captured graph per slot and layer)
                                                              -> event done[k]
    copy-out stream  wait done[k]; D2H output of step k       -> event out_done[k]

A slot is reused only after its previous decode has consumed its inputs
(copy-in waits done[k - depth]) and its previous output has left the device
(compute waits out_done[k - depth]).  Torch provides the memory, streams and
events; every step of the computation is the library's kernel.
"""

from __future__ import annotations

from typing import List, Optional

import torch

from . import _binding as b


class DecodePipeline:
    """Double-buffered (``depth`` slots) decode steps with host inputs and outputs.

    ``submit`` enqueues one step and returns at once with the event that marks
    its output in ``h_out``; the caller keeps ``h_q``, ``h_block_table``,
    ``h_seq_lens`` unchanged and does not read ``h_out`` before that event.
    Host tensors should be pinned for the copies to be asynchronous.
    """

    def __init__(self, k_cache, v_cache, num_seqs: int, num_heads: int, max_blocks: int, scale: float,
                 max_seq_len: int, partition_size: int = 0, depth: int = 2, use_graph: bool = True):
        """``k_cache`` / ``v_cache``: one layer's paged cache, or a list with one per layer
        (``submit(..., layer=i)`` picks one; all layers share shape and dtype)."""
        if depth < 1:
            raise ValueError("depth must be >= 1")
        ks = list(k_cache) if isinstance(k_cache, (list, tuple)) else [k_cache]
        vs = list(v_cache) if isinstance(v_cache, (list, tuple)) else [v_cache]
        if not ks or len(ks) != len(vs):
            raise ValueError("k_cache and v_cache must hold the same number of layers")
        for i, (kc, vc) in enumerate(zip(ks, vs)):
            b._cuda(f"k_cache[{i}]", kc, dtype=ks[0].dtype, ndim=4)
            b._cuda(f"v_cache[{i}]", vc, dtype=ks[0].dtype, ndim=4)
            if kc.shape != ks[0].shape or vc.shape != ks[0].shape:
                raise ValueError("every layer's cache must have one shape")
        dev = ks[0].device
        D = ks[0].shape[3]
        self.k_caches, self.v_caches = ks, vs
        self.scale, self.max_seq_len, self.partition_size = float(scale), int(max_seq_len), int(partition_size)
        self.depth = depth
        self.q = [torch.empty(num_seqs, num_heads, D, dtype=ks[0].dtype, device=dev) for _ in range(depth)]
        self.bt = [torch.empty(num_seqs, max_blocks, dtype=torch.int32, device=dev) for _ in range(depth)]
        self.sl = [torch.empty(num_seqs, dtype=torch.int32, device=dev) for _ in range(depth)]
        self.out = [torch.empty_like(self.q[0]) for _ in range(depth)]
        need = b.metis_decode_workspace_bytes(num_seqs, num_heads, D, max_seq_len, partition_size)
        self.ws = [torch.empty(max(need, 256), dtype=torch.uint8, device=dev) for _ in range(depth)]
        self.copy_in = torch.cuda.Stream(device=dev)
        self.compute = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)
        self.in_done: List[torch.cuda.Event] = [torch.cuda.Event() for _ in range(depth)]
        self.done: List[torch.cuda.Event] = [torch.cuda.Event() for _ in range(depth)]
        self.out_done: List[torch.cuda.Event] = [torch.cuda.Event() for _ in range(depth)]
        self.k = 0
        self.graphs: Optional[List[List[torch.cuda.CUDAGraph]]] = None
        if use_graph:
            self._capture()

    def _decode(self, s: int, layer: int) -> None:
        b.metis_paged_attn_decode(self.q[s], self.k_caches[layer], self.v_caches[layer], self.bt[s], self.sl[s],
                                  self.scale, out=self.out[s], partition_size=self.partition_size,
                                  max_seq_len=self.max_seq_len, workspace=self.ws[s])

    def _capture(self) -> None:
        # one eager call per slot on zeroed inputs (lengths 0: nothing is read), then capture
        for s in range(self.depth):
            self.q[s].zero_()
            self.bt[s].fill_(-1)
            self.sl[s].zero_()
        with torch.cuda.stream(self.compute):
            for s in range(self.depth):
                self._decode(s, 0)
        self.compute.synchronize()
        self.graphs = []   # [slot][layer]
        for s in range(self.depth):
            per_layer = []
            for layer in range(len(self.k_caches)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.compute):
                    self._decode(s, layer)
                per_layer.append(g)
            self.graphs.append(per_layer)
        self.compute.synchronize()
        b.metis_read_status(clear=True)

    def submit(self, h_q: torch.Tensor, h_block_table: torch.Tensor, h_seq_lens: torch.Tensor,
               h_out: torch.Tensor, layer: int = 0) -> torch.cuda.Event:
        """Enqueue one decode step over layer ``layer``'s cache: host inputs in, output to
        ``h_out``; returns its completion event."""
        if not 0 <= layer < len(self.k_caches):
            raise IndexError(f"layer {layer} out of range ({len(self.k_caches)} layers)")
        s = self.k % self.depth
        if self.k >= self.depth:
            self.copy_in.wait_event(self.done[s])       # the slot's inputs were consumed
            self.compute.wait_event(self.out_done[s])   # the slot's output has left the device
        with torch.cuda.stream(self.copy_in):
            self.q[s].copy_(h_q, non_blocking=True)
            self.bt[s].copy_(h_block_table, non_blocking=True)
            self.sl[s].copy_(h_seq_lens, non_blocking=True)
            self.in_done[s].record(self.copy_in)
        self.compute.wait_event(self.in_done[s])
        if self.graphs is not None:
            with torch.cuda.stream(self.compute):
                self.graphs[s][layer].replay()
        else:
            with torch.cuda.stream(self.compute):
                self._decode(s, layer)
        self.done[s].record(self.compute)
        self.copy_out.wait_event(self.done[s])
        with torch.cuda.stream(self.copy_out):
            h_out.copy_(self.out[s], non_blocking=True)
            self.out_done[s].record(self.copy_out)
        self.k += 1
        return self.out_done[s]

    def synchronize(self) -> None:
        for st in (self.copy_in, self.compute, self.copy_out):
            st.synchronize()
