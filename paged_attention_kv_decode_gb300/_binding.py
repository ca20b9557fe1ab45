"""ctypes binding of ``libmetis_attn.so`` -- argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but check the torch tensors it is handed (device, dtype, shape,
contiguity), allocate outputs / workspace with torch when the caller did not
pass them, and hand raw device pointers plus the current CUDA stream to the
library.  All computation happens in the library's CUDA kernels; there is no
CPU or PyTorch fallback: a missing library or a CPU tensor raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libmetis_attn.so")

METIS_F32 = 0
METIS_BF16 = 1

STATUS_BAD_BLOCK_ID = 1
STATUS_SEQ_TOO_LONG = 2
STATUS_WAIT_TIMEOUT = 4
STATUS_BAD_Q_LEN = 8
STATUS_TABLE_FULL = 16
STATUS_OUT_OF_PAGES = 32
STATUS_BAD_OFFSETS = 64

_ERRORS = {
    -1: "METIS_E_NULL",
    -2: "METIS_E_SHAPE",
    -3: "METIS_E_UNSUPPORTED",
    -4: "METIS_E_ALIGN",
    -5: "METIS_E_WORKSPACE",
    -6: "METIS_E_CUDA",
}


class MetisError(RuntimeError):
    """A non-zero status from the library; ``code`` is the METIS_E_* value."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{_ERRORS.get(code, code)}: {message}")
        self.code = code


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_f = ctypes.c_float

# name -> (restype, argtypes); mirrors include/metis_attn.h
SIGNATURES = {
    "metis_paged_attn_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                     _vp, _sz, _vp]),
    "metis_paged_attn_decode_partials": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                              _vp, _sz, _vp]),
    "metis_paged_attn_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                                             _i, _i, _vp]),
    "metis_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "metis_paged_attn_prefill_chunk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                                            _i, _f, _i, _vp, _sz, _vp]),
    "metis_prefill_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "metis_mla_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "metis_mla_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "metis_merge_attn_states": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "metis_read_status": (_i, [ctypes.POINTER(ctypes.c_uint32), _i]),
    "metis_last_error": (ctypes.c_char_p, []),
    "metis_version": (_i, []),
    "metis_reshape_and_cache": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "metis_mla_reshape_and_cache": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "metis_prefix_block_hashes": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "metis_prefix_table_init": (_i, [_vp, _vp, _vp, _i, _vp]),
    "metis_prefix_lookup_workspace_bytes": (_sz, [_i]),
    "metis_prefix_lookup": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "metis_debug_wait_probe": (_i, [ctypes.c_uint64, _vp]),
}


def load_library(path: str = LIB_PATH):
    """Load the library once (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not found at {path}: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        raise MetisError(rc, load_library().metis_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return METIS_F32
    if dt == torch.bfloat16:
        return METIS_BF16
    raise TypeError(f"unsupported dtype {dt}; use float32 or bfloat16")


def _cuda(name: str, t: torch.Tensor, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def metis_version() -> int:
    return load_library().metis_version()


def metis_last_error() -> str:
    return load_library().metis_last_error().decode()


def metis_read_status(clear: bool = True) -> int:
    """The device status word (METIS_STATUS_* bits); synchronises the device."""
    v = ctypes.c_uint32(0)
    _check(load_library().metis_read_status(ctypes.byref(v), int(bool(clear))))
    return int(v.value)


def metis_decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_seq_len: int,
                                 partition_size: int) -> int:
    return int(load_library().metis_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_seq_len,
                                                           partition_size))


def metis_paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                            out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                            partition_size: int = 0, max_seq_len: Optional[int] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None,
                            want_lse: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Paged decode; returns ``(out, lse_out)``.  ``max_seq_len=None`` reads seq_lens (a sync)."""
    lib = load_library()
    _cuda("q", q, ndim=3)
    dt = _dtype_code(q.dtype)
    _cuda("k_cache", k_cache, dtype=q.dtype, ndim=4)
    _cuda("v_cache", v_cache, dtype=q.dtype, ndim=4)
    _cuda("block_table", block_table, dtype=torch.int32, ndim=2)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    S, H, D = q.shape
    nb, bs, G, Dk = k_cache.shape
    if v_cache.shape != k_cache.shape or Dk != D or block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, dtype=q.dtype, ndim=3)
    if lse_out is None and want_lse:
        lse_out = torch.empty((S, H), dtype=torch.float32, device=q.device)
    if lse_out is not None:
        _cuda("lse_out", lse_out, dtype=torch.float32, ndim=2)
    if max_seq_len is None:
        max_seq_len = max(1, int(seq_lens.max().item())) if S else 1
    need = metis_decode_workspace_bytes(S, H, D, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.metis_paged_attn_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse_out),
        S, H, G, D, bs, block_table.shape[1], nb, dt, float(scale), int(partition_size), int(max_seq_len),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse_out


def metis_merge_attn_states(part_out: torch.Tensor, part_lse: torch.Tensor, seq_lens: torch.Tensor,
                            partition_size: int, *, out: Optional[torch.Tensor] = None,
                            lse_out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                            stream=None, want_lse: bool = False):
    """Log-sum-exp merge of ``part_out`` [S, H, P, D] / ``part_lse`` [S, H, P]; returns ``(out, lse_out)``."""
    lib = load_library()
    _cuda("part_out", part_out, dtype=torch.float32, ndim=4)
    _cuda("part_lse", part_lse, dtype=torch.float32, ndim=3)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    S, H, P, D = part_out.shape
    if part_lse.shape != (S, H, P) or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((S, H, D), dtype=out_dtype, device=part_out.device)
    _cuda("out", out, ndim=3)
    if lse_out is None and want_lse:
        lse_out = torch.empty((S, H), dtype=torch.float32, device=part_out.device)
    _check(lib.metis_merge_attn_states(_ptr(part_out), _ptr(part_lse), _ptr(seq_lens), int(partition_size),
                                       _ptr(out), _ptr(lse_out), S, H, D, P, _dtype_code(out.dtype),
                                       _stream(stream)))
    return out, lse_out


def split_workspace_views(workspace: torch.Tensor, num_seqs: int, num_heads: int, head_dim: int, max_seq_len: int,
                          partition_size: int):
    """``(part_out, part_lse)`` views of a split-KV decode workspace (the layout the header documents)."""
    parts = -(-max_seq_len // partition_size)
    units = num_seqs * num_heads * parts
    off = -(-units * head_dim * 4 // 256) * 256
    flat = workspace.view(torch.uint8)
    part_out = flat[:units * head_dim * 4].view(torch.float32).view(num_seqs, num_heads, parts, head_dim)
    part_lse = flat[off:off + units * 4].view(torch.float32).view(num_seqs, num_heads, parts)
    return part_out, part_lse


def metis_paged_attn_decode_partials(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                     block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                                     partition_size: int, max_seq_len: int, workspace: Optional[torch.Tensor] = None,
                                     stream=None) -> torch.Tensor:
    """Split-KV partials into ``workspace`` (allocated when None); returns the workspace."""
    lib = load_library()
    _cuda("q", q, ndim=3)
    dt = _dtype_code(q.dtype)
    _cuda("k_cache", k_cache, dtype=q.dtype, ndim=4)
    _cuda("v_cache", v_cache, dtype=q.dtype, ndim=4)
    _cuda("block_table", block_table, dtype=torch.int32, ndim=2)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    S, H, D = q.shape
    nb, bs, G, _ = k_cache.shape
    need = metis_decode_workspace_bytes(S, H, D, max_seq_len, partition_size)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.metis_paged_attn_decode_partials(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), S, H, G, D, bs,
        block_table.shape[1], nb, dt, float(scale), int(partition_size), int(max_seq_len), _ptr(workspace), ws_bytes,
        _stream(stream)))
    return workspace


NOALLOC_SCRATCH_BYTES = 64 << 20


def metis_paged_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                    block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                                    out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                                    partition_size: int = 0, max_seq_len: int, stream=None):
    """Paged decode whose split-KV scratch is the library's static device array.

    For callers that cannot allocate device memory: this wrapper allocates
    nothing either, so ``out`` (and ``lse_out`` if wanted) must be passed in
    and ``max_seq_len`` must be given.  Calls that overlap on the GPU share
    the one scratch array and race; calls on one stream are ordered.
    """
    lib = load_library()
    _cuda("q", q, ndim=3)
    dt = _dtype_code(q.dtype)
    _cuda("k_cache", k_cache, dtype=q.dtype, ndim=4)
    _cuda("v_cache", v_cache, dtype=q.dtype, ndim=4)
    _cuda("block_table", block_table, dtype=torch.int32, ndim=2)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    _cuda("out", out, dtype=q.dtype, ndim=3)
    if lse_out is not None:
        _cuda("lse_out", lse_out, dtype=torch.float32, ndim=2)
    S, H, D = q.shape
    nb, bs, G, _ = k_cache.shape
    _check(lib.metis_paged_attn_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse_out),
        S, H, G, D, bs, block_table.shape[1], nb, dt, float(scale), int(partition_size), int(max_seq_len),
        _stream(stream)))
    return out, lse_out


def metis_prefill_workspace_bytes(num_seqs: int, num_tokens: int, num_heads: int, num_kv_heads: int) -> int:
    return int(load_library().metis_prefill_workspace_bytes(num_seqs, num_tokens, num_heads, num_kv_heads))


def metis_paged_attn_prefill_chunk(q: torch.Tensor, cu_q_lens: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                                   scale: float, *, out: Optional[torch.Tensor] = None,
                                   lse_out: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
                                   workspace: Optional[torch.Tensor] = None, stream=None, want_lse: bool = False):
    """Chunked prefill (+ single-token decodes); returns ``(out, lse_out)``."""
    lib = load_library()
    _cuda("q", q, ndim=3)
    dt = _dtype_code(q.dtype)
    _cuda("cu_q_lens", cu_q_lens, dtype=torch.int32, ndim=1)
    _cuda("k_cache", k_cache, dtype=q.dtype, ndim=4)
    _cuda("v_cache", v_cache, dtype=q.dtype, ndim=4)
    _cuda("block_table", block_table, dtype=torch.int32, ndim=2)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    T, H, D = q.shape
    nb, bs, G, Dk = k_cache.shape
    S = seq_lens.shape[0]
    if cu_q_lens.shape[0] != S + 1 or block_table.shape[0] != S or Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, dtype=q.dtype, ndim=3)
    if lse_out is None and want_lse:
        lse_out = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse_out is not None:
        _cuda("lse_out", lse_out, dtype=torch.float32, ndim=2)
    if max_seq_len is None:
        max_seq_len = max(1, int(seq_lens.max().item())) if S else 1
    need = metis_prefill_workspace_bytes(S, T, H, G)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.metis_paged_attn_prefill_chunk(
        _ptr(q), _ptr(cu_q_lens), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out),
        _ptr(lse_out), S, T, H, G, D, bs, block_table.shape[1], nb, dt, float(scale), int(max_seq_len),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse_out


def metis_mla_workspace_bytes(num_seqs: int, num_heads: int, max_seq_len: int, partition_size: int) -> int:
    return int(load_library().metis_mla_workspace_bytes(num_seqs, num_heads, max_seq_len, partition_size))


def metis_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                     scale: float, *, d_latent: int = 512, out: Optional[torch.Tensor] = None,
                     lse_out: Optional[torch.Tensor] = None, partition_size: int = 0,
                     max_seq_len: Optional[int] = None, workspace: Optional[torch.Tensor] = None, stream=None,
                     want_lse: bool = False):
    """MLA decode over a paged latent cache; returns ``(out, lse_out)``."""
    lib = load_library()
    _cuda("q", q, dtype=torch.bfloat16, ndim=3)
    _cuda("kv_cache", kv_cache, dtype=torch.bfloat16, ndim=3)
    _cuda("block_table", block_table, dtype=torch.int32, ndim=2)
    _cuda("seq_lens", seq_lens, dtype=torch.int32, ndim=1)
    S, H, dq = q.shape
    nb, bs, dk = kv_cache.shape
    if dk != dq or block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((S, H, d_latent), dtype=q.dtype, device=q.device)
    _cuda("out", out, dtype=q.dtype, ndim=3)
    if lse_out is None and want_lse:
        lse_out = torch.empty((S, H), dtype=torch.float32, device=q.device)
    if lse_out is not None:
        _cuda("lse_out", lse_out, dtype=torch.float32, ndim=2)
    if max_seq_len is None:
        max_seq_len = max(1, int(seq_lens.max().item())) if S else 1
    need = metis_mla_workspace_bytes(S, H, max_seq_len, partition_size)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.metis_mla_decode(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(out),
                                _ptr(lse_out), S, H, d_latent, dq - d_latent, bs, block_table.shape[1], nb,
                                float(scale), int(partition_size), int(max_seq_len), _ptr(workspace), ws_bytes,
                                _stream(stream)))
    return out, lse_out


def metis_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            slot_mapping: torch.Tensor, stream=None) -> None:
    """Write ``key`` / ``value`` rows ``[N, G, D]`` into the paged caches ``[nb, bs, G, D]``
    at ``slot_mapping`` (int64 ``[N]``, negative = padding); in place, asynchronous."""
    lib = load_library()
    _cuda("key", key, ndim=3)
    dt = key.dtype
    _cuda("value", value, dtype=dt, ndim=3)
    _cuda("k_cache", k_cache, dtype=dt, ndim=4)
    _cuda("v_cache", v_cache, dtype=dt, ndim=4)
    _cuda("slot_mapping", slot_mapping, dtype=torch.int64, ndim=1)
    N, G, D = key.shape
    nb, bs = k_cache.shape[:2]
    if (value.shape != key.shape or tuple(k_cache.shape[2:]) != (G, D) or v_cache.shape != k_cache.shape
            or slot_mapping.shape[0] != N):
        raise ValueError("inconsistent shapes")
    _check(lib.metis_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                       N, G, D, bs, nb, _dtype_code(dt), _stream(stream)))


def metis_mla_reshape_and_cache(kv_c: torch.Tensor, k_pe: torch.Tensor, kv_cache: torch.Tensor,
                                slot_mapping: torch.Tensor, stream=None) -> None:
    """Write rows ``[kv_c | k_pe]`` (bf16 ``[N, d_latent]``, ``[N, d_rope]``) into the latent
    cache ``[nb, bs, d_latent + d_rope]`` at ``slot_mapping``; in place, asynchronous."""
    lib = load_library()
    _cuda("kv_c", kv_c, dtype=torch.bfloat16, ndim=2)
    _cuda("k_pe", k_pe, dtype=torch.bfloat16, ndim=2)
    _cuda("kv_cache", kv_cache, dtype=torch.bfloat16, ndim=3)
    _cuda("slot_mapping", slot_mapping, dtype=torch.int64, ndim=1)
    N, dl = kv_c.shape
    dr = k_pe.shape[1]
    nb, bs, dk = kv_cache.shape
    if k_pe.shape[0] != N or dk != dl + dr or slot_mapping.shape[0] != N:
        raise ValueError("inconsistent shapes")
    _check(lib.metis_mla_reshape_and_cache(_ptr(kv_c), _ptr(k_pe), _ptr(kv_cache), _ptr(slot_mapping), N, dl, dr,
                                           bs, nb, _stream(stream)))


def metis_prefix_block_hashes(token_ids: torch.Tensor, cu_tokens: torch.Tensor, cu_pages: torch.Tensor,
                              block_size: int, total_pages: int, keys_out: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """Chained key of every full page (int64 ``[total_pages]`` holding the uint64 bit
    pattern).  ``cu_pages`` (int32 ``[S + 1]``) and ``total_pages`` are the caller's:
    sequence s has ``(cu_tokens[s+1] - cu_tokens[s]) // block_size`` keys."""
    lib = load_library()
    _cuda("token_ids", token_ids, dtype=torch.int32, ndim=1)
    _cuda("cu_tokens", cu_tokens, dtype=torch.int32, ndim=1)
    _cuda("cu_pages", cu_pages, dtype=torch.int32, ndim=1)
    S = cu_tokens.shape[0] - 1
    if cu_pages.shape[0] != S + 1:
        raise ValueError("cu_tokens and cu_pages must both have num_seqs + 1 entries")
    if keys_out is None:
        keys_out = torch.empty(total_pages, dtype=torch.int64, device=token_ids.device)
    _cuda("keys_out", keys_out, dtype=torch.int64, ndim=1)
    if keys_out.shape[0] < total_pages:
        raise ValueError("keys_out is shorter than total_pages")
    _check(lib.metis_prefix_block_hashes(_ptr(token_ids), _ptr(cu_tokens), _ptr(cu_pages), S, int(block_size),
                                         int(total_pages), _ptr(keys_out), _stream(stream)))
    return keys_out


def metis_prefix_table_init(table_keys: torch.Tensor, table_pages: torch.Tensor, table_claim: torch.Tensor,
                            stream=None) -> None:
    """Empty the open-addressing table (int64 keys, int32 pages, int32 claim; one
    power-of-two capacity); asynchronous."""
    lib = load_library()
    _cuda("table_keys", table_keys, dtype=torch.int64, ndim=1)
    _cuda("table_pages", table_pages, dtype=torch.int32, ndim=1)
    _cuda("table_claim", table_claim, dtype=torch.int32, ndim=1)
    cap = table_keys.shape[0]
    if table_pages.shape[0] != cap or table_claim.shape[0] != cap:
        raise ValueError("the three table arrays must have one capacity")
    _check(lib.metis_prefix_table_init(_ptr(table_keys), _ptr(table_pages), _ptr(table_claim), cap,
                                       _stream(stream)))


def prefix_table_alloc(capacity: int, device="cuda", stream=None):
    """Allocate and empty a table of ``capacity`` slots; returns ``(keys, pages, claim)``."""
    keys = torch.empty(capacity, dtype=torch.int64, device=device)
    pages = torch.empty(capacity, dtype=torch.int32, device=device)
    claim = torch.empty(capacity, dtype=torch.int32, device=device)
    metis_prefix_table_init(keys, pages, claim, stream)
    return keys, pages, claim


def metis_prefix_lookup_workspace_bytes(n: int) -> int:
    return int(load_library().metis_prefix_lookup_workspace_bytes(n))


def metis_prefix_lookup(keys: torch.Tensor, table, free_stack: torch.Tensor, free_count: torch.Tensor,
                        refcount: torch.Tensor, pages_out: Optional[torch.Tensor] = None,
                        hits_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None):
    """Lookup-or-allocate of ``keys`` (int64 ``[n]``) in ``table`` (the tuple of
    ``prefix_table_alloc``); ``free_stack`` int32 (top at the end), ``free_count``
    int32 ``[1]`` and ``refcount`` int32 ``[num_pages]`` are updated in place.
    Returns ``(pages int32 [n], hits uint8 [n])``; asynchronous."""
    lib = load_library()
    table_keys, table_pages, table_claim = table
    _cuda("keys", keys, dtype=torch.int64, ndim=1)
    _cuda("table_keys", table_keys, dtype=torch.int64, ndim=1)
    _cuda("table_pages", table_pages, dtype=torch.int32, ndim=1)
    _cuda("table_claim", table_claim, dtype=torch.int32, ndim=1)
    _cuda("free_stack", free_stack, dtype=torch.int32, ndim=1)
    _cuda("free_count", free_count, dtype=torch.int32, ndim=1)
    _cuda("refcount", refcount, dtype=torch.int32, ndim=1)
    n = keys.shape[0]
    dev = keys.device
    if pages_out is None:
        pages_out = torch.empty(n, dtype=torch.int32, device=dev)
    if hits_out is None:
        hits_out = torch.empty(n, dtype=torch.uint8, device=dev)
    _cuda("pages_out", pages_out, dtype=torch.int32, ndim=1)
    _cuda("hits_out", hits_out, dtype=torch.uint8, ndim=1)
    if pages_out.shape[0] < n or hits_out.shape[0] < n:
        raise ValueError("pages_out / hits_out are shorter than keys")
    need = metis_prefix_lookup_workspace_bytes(n)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _cuda("workspace", workspace, dtype=torch.uint8, ndim=1)
    cap = table_keys.shape[0]
    _check(lib.metis_prefix_lookup(_ptr(keys), n, _ptr(table_keys), _ptr(table_pages), _ptr(table_claim), cap,
                                   _ptr(free_stack), free_stack.shape[0], _ptr(free_count), _ptr(refcount),
                                   refcount.shape[0], _ptr(pages_out), _ptr(hits_out), _ptr(workspace),
                                   workspace.numel(), _stream(stream)))
    return pages_out, hits_out


def metis_debug_wait_probe(limit_ns: int, stream=None) -> None:
    """Run the bounded-wait give-up path once (a wait that nothing completes, limited to limit_ns)."""
    _check(load_library().metis_debug_wait_probe(int(limit_ns), _stream(stream)))
