"""The C ABI: every declared symbol is exported, and bad arguments are rejected on the host.

These tests run without a GPU.  Every call below is one the library must
reject before touching CUDA, so nothing is ever launched with the fake
pointers used here.
"""

import ctypes
import os
import re

import pytest

import paged_attention_kv_decode_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for fname in sorted(os.listdir(HEADER_DIR)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(metis_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pa.LIB_PATH):
        from paged_attention_kv_decode_gb300 import build
        build.build()
    return pa.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("metis_paged_attn_decode", "metis_paged_attn_decode_partials", "metis_merge_attn_states", "metis_decode_workspace_bytes",
              "metis_read_status", "metis_last_error", "metis_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_covers_every_declared_symbol():
    assert sorted(pa.SIGNATURES) == declared_functions()


def test_version(lib):
    assert pa.metis_version() >= 100


def test_workspace_bytes(lib):
    assert pa.metis_decode_workspace_bytes(4, 8, 128, 1000, 0) == 0
    n = pa.metis_decode_workspace_bytes(4, 8, 128, 1000, 512)   # 2 partitions
    units = 4 * 8 * 2
    assert n >= units * 128 * 4 + units * 4 and n % 256 == 0


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced: every call below is rejected first


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, out=FAKE, lse=None, S=4, H=32, G=8, D=128, bs=16,
             max_blocks=8, num_blocks=64, dtype=pa.METIS_BF16, scale=0.088, P=0, max_len=128, ws=None,
             ws_bytes=0, stream=None)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.metis_paged_attn_decode(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["bt"]), vp(a["sl"]), vp(a["out"]),
                                       vp(a["lse"]), a["S"], a["H"], a["G"], a["D"], a["bs"], a["max_blocks"],
                                       a["num_blocks"], a["dtype"], a["scale"], a["P"], a["max_len"], vp(a["ws"]),
                                       a["ws_bytes"], vp(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(bt=None), -1), (dict(out=None), -1),
    (dict(S=-1), -2), (dict(H=0), -2), (dict(max_len=0), -2), (dict(num_blocks=0), -2),
    (dict(H=30), -2),                                   # not a multiple of kv heads
    (dict(D=96), -3), (dict(bs=8), -3), (dict(dtype=7), -3),
    (dict(H=48, G=4), -3),                              # ratio 12 > 8
    (dict(H=24, G=8), -3),                              # bf16 ratio 3
    (dict(q=FAKE + 2), -4), (dict(k=FAKE + 8), -4), (dict(sl=FAKE + 1), -4),
    (dict(P=100), -2), (dict(P=-16), -2),
    (dict(P=512, max_len=100_000), -5),                 # split needs a workspace
    (dict(P=512, ws=FAKE, ws_bytes=16), -5),            # too small
    (dict(scale=float("nan")), -2),
    (dict(max_blocks=1 << 28, bs=64), -2),              # max_blocks * bs overflows int32
    (dict(S=70000), -2),
])
def test_decode_rejects(lib, kw, code):
    assert _decode(lib, **kw) == code
    assert pa.metis_last_error() != ""


def test_decode_empty_batch_is_a_no_op(lib):
    assert _decode(lib, S=0) == 0
    assert pa.metis_last_error() == ""


@pytest.mark.parametrize("kw,code", [
    (dict(po=None), -1), (dict(D=130), -3), (dict(D=1024), -3), (dict(P=0), -2), (dict(dt=3), -3),
    (dict(po=FAKE + 4), -4),
])
def test_merge_rejects(lib, kw, code):
    a = dict(po=FAKE, pl=FAKE, sl=FAKE, P=512, out=FAKE, lse=None, S=2, H=4, D=128, maxp=3, dt=pa.METIS_BF16)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = lib.metis_merge_attn_states(vp(a["po"]), vp(a["pl"]), vp(a["sl"]), a["P"], vp(a["out"]), vp(a["lse"]),
                                     a["S"], a["H"], a["D"], a["maxp"], a["dt"], None)
    assert rc == code


def test_read_status_rejects_null(lib):
    assert lib.metis_read_status(None, 0) == -1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 4, 64)
    kc = torch.zeros(2, 16, 1, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.metis_paged_attn_decode(q, kc, kc, torch.zeros(1, 1, dtype=torch.int32),
                                   torch.ones(1, dtype=torch.int32), 0.1, max_seq_len=1)


def test_partials_reject(lib):
    vp = ctypes.c_void_p
    f = lib.metis_paged_attn_decode_partials
    # partition_size 0 is meaningless for partials
    assert f(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 4, 32, 8, 128, 16, 8, 64, pa.METIS_BF16, 0.1, 0, 128,
             vp(FAKE), 1 << 20, None) == -2
    # workspace too small
    assert f(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 4, 32, 8, 128, 16, 8, 64, pa.METIS_BF16, 0.1, 64, 128,
             vp(FAKE), 64, None) == -5


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(cu=None), -1),
    (dict(dtype=0), -3), (dict(D=96), -3), (dict(bs=8), -3), (dict(H=24, G=8), -3), (dict(H=30), -2),
    (dict(q=FAKE + 8), -4), (dict(cu=FAKE + 2), -4),
    (dict(ws=None), -5), (dict(ws_bytes=16), -5), (dict(ws=FAKE + 16), -5),
    (dict(T=-1), -2), (dict(max_len=0), -2),
])
def test_prefill_rejects(lib, kw, code):
    a = dict(q=FAKE, cu=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, out=FAKE, lse=None, S=4, T=100, H=32, G=8, D=128,
             bs=16, max_blocks=8, num_blocks=64, dtype=pa.METIS_BF16, scale=0.088, max_len=128, ws=FAKE,
             ws_bytes=1 << 20)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = lib.metis_paged_attn_prefill_chunk(vp(a["q"]), vp(a["cu"]), vp(a["k"]), vp(a["v"]), vp(a["bt"]),
                                            vp(a["sl"]), vp(a["out"]), vp(a["lse"]), a["S"], a["T"], a["H"], a["G"],
                                            a["D"], a["bs"], a["max_blocks"], a["num_blocks"], a["dtype"], a["scale"],
                                            a["max_len"], vp(a["ws"]), a["ws_bytes"], None)
    assert rc == code


def test_prefill_workspace_bytes(lib):
    # 4 heads per group -> 32-token query tiles, computed in pairs: ceil(100 / 64) + 4 sequences = 6 items
    # of 16 bytes + a 256-byte header
    assert pa.metis_prefill_workspace_bytes(4, 100, 32, 8) == 256 + 6 * 16
    assert pa.metis_prefill_workspace_bytes(0, 100, 32, 8) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(kv=None), -1), (dict(dl=256), -3), (dict(dr=32), -3), (dict(H=100), -3),
    (dict(bs=8), -3), (dict(P=48), -2), (dict(q=FAKE + 4), -4), (dict(ws=None), -5), (dict(ws_bytes=8), -5),
    (dict(S=-2), -2),
])
def test_mla_rejects(lib, kw, code):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, out=FAKE, lse=None, S=4, H=128, dl=512, dr=64, bs=64,
             max_blocks=8, num_blocks=64, scale=0.07, P=256, max_len=512, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    rc = lib.metis_mla_decode(vp(a["q"]), vp(a["kv"]), vp(a["bt"]), vp(a["sl"]), vp(a["out"]), vp(a["lse"]), a["S"],
                              a["H"], a["dl"], a["dr"], a["bs"], a["max_blocks"], a["num_blocks"], a["scale"], a["P"],
                              a["max_len"], vp(a["ws"]), a["ws_bytes"], None)
    assert rc == code


def test_mla_workspace_bytes(lib):
    assert pa.metis_mla_workspace_bytes(4, 128, 512, 0) > 0
    n = pa.metis_mla_workspace_bytes(4, 128, 512, 256)       # 2 partitions of fp32 partials
    assert n >= 4 * 128 * 2 * 512 * 4


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -2), (dict(key=None), -1), (dict(slots=None), -1), (dict(dt=3), -3),
    (dict(G=1, D=4, dt=pa.METIS_BF16), -3),                 # 8-byte rows cannot be copied as 16-byte vectors
    (dict(key=FAKE + 8), -4), (dict(slots=FAKE + 4), -4), (dict(G=0), -2), (dict(nb=0), -2),
])
def test_reshape_and_cache_rejects(lib, kw, code):
    a = dict(key=FAKE, value=FAKE, kc=FAKE, vc=FAKE, slots=FAKE, n=16, G=8, D=128, bs=16, nb=64, dt=pa.METIS_BF16)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.metis_reshape_and_cache(vp(a["key"]), vp(a["value"]), vp(a["kc"]), vp(a["vc"]), vp(a["slots"]), a["n"],
                                     a["G"], a["D"], a["bs"], a["nb"], a["dt"], None)
    assert rc == code


def test_reshape_and_cache_empty_is_a_no_op(lib):
    vp = ctypes.c_void_p
    assert lib.metis_reshape_and_cache(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0, 8, 128, 16, 64,
                                       pa.METIS_BF16, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -2), (dict(kv_c=None), -1), (dict(dl=500), -3), (dict(dr=0), -2), (dict(kv=FAKE + 8), -4),
])
def test_mla_reshape_and_cache_rejects(lib, kw, code):
    a = dict(kv_c=FAKE, k_pe=FAKE, kv=FAKE, slots=FAKE, n=16, dl=512, dr=64, bs=64, nb=32)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.metis_mla_reshape_and_cache(vp(a["kv_c"]), vp(a["k_pe"]), vp(a["kv"]), vp(a["slots"]), a["n"], a["dl"],
                                         a["dr"], a["bs"], a["nb"], None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(S=-1), -2), (dict(total=-1), -2), (dict(tok=None), -1), (dict(keys=None), -1), (dict(bs=0), -2),
    (dict(tok=FAKE + 2), -4), (dict(cup=FAKE + 1), -4), (dict(keys=FAKE + 4), -4),
])
def test_prefix_block_hashes_rejects(lib, kw, code):
    a = dict(tok=FAKE, cut=FAKE, cup=FAKE, S=4, bs=16, total=8, keys=FAKE)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.metis_prefix_block_hashes(vp(a["tok"]), vp(a["cut"]), vp(a["cup"]), a["S"], a["bs"], a["total"],
                                       vp(a["keys"]), None)
    assert rc == code, pa.metis_last_error()


def test_prefix_block_hashes_empty_is_a_no_op(lib):
    vp = ctypes.c_void_p
    assert lib.metis_prefix_block_hashes(vp(FAKE), vp(FAKE), vp(FAKE), 0, 16, 8, vp(FAKE), None) == 0
    assert lib.metis_prefix_block_hashes(None, None, None, 4, 16, 0, None, None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(cap=0), -2), (dict(cap=6), -2), (dict(keys=None), -1), (dict(keys=FAKE + 4), -4), (dict(claim=FAKE + 2), -4),
])
def test_prefix_table_init_rejects(lib, kw, code):
    a = dict(keys=FAKE, pages=FAKE, claim=FAKE, cap=1024)
    a.update(kw)
    vp = ctypes.c_void_p
    assert lib.metis_prefix_table_init(vp(a["keys"]), vp(a["pages"]), vp(a["claim"]), a["cap"], None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -2), (dict(keys=None), -1), (dict(fc=None), -1), (dict(cap=100), -2), (dict(fcap=-1), -2),
    (dict(npages=0), -2), (dict(keys=FAKE + 4), -4), (dict(po=FAKE + 2), -4), (dict(ws=None), -5),
    (dict(ws_bytes=256), -5), (dict(ws=FAKE + 16), -5),
])
def test_prefix_lookup_rejects(lib, kw, code):
    a = dict(keys=FAKE, n=16, tk=FAKE, tp=FAKE, tc=FAKE, cap=1024, fs=FAKE, fcap=64, fc=FAKE, rc=FAKE, npages=64,
             po=FAKE, ho=FAKE, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.metis_prefix_lookup(vp(a["keys"]), a["n"], vp(a["tk"]), vp(a["tp"]), vp(a["tc"]), a["cap"], vp(a["fs"]),
                                 a["fcap"], vp(a["fc"]), vp(a["rc"]), a["npages"], vp(a["po"]), vp(a["ho"]),
                                 vp(a["ws"]), a["ws_bytes"], None)
    assert rc == code, pa.metis_last_error()


def test_prefix_lookup_empty_and_workspace(lib):
    assert lib.metis_prefix_lookup(None, 0, None, None, None, 0, None, 0, None, None, 0, None, None, None, 0, None) == 0
    assert lib.metis_prefix_lookup_workspace_bytes(0) == 0
    assert lib.metis_prefix_lookup_workspace_bytes(16) >= 16 * 5


@pytest.mark.parametrize("limit_ns", [0, 1_000_000_001, 2 ** 63])
def test_wait_probe_rejects_limits_outside_one_second(lib, limit_ns):
    assert lib.metis_debug_wait_probe(limit_ns, None) == -2   # METIS_E_SHAPE
    assert "limit_ns" in pa.metis_last_error()
