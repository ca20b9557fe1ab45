"""Shared test helpers: device transfer, tolerance checks, block re-placement."""

import numpy as np
import torch

# Tolerances of the parity bar: fp32 max |d| <= 1e-5; bf16 inputs with fp32
# accumulation |d| <= 1.5e-2 + 1e-2 |ref| elementwise.  lse (always fp32) of a
# bf16 case is held to 1e-3 absolute: it only sees fp32 rounding of exact
# bf16 products -- except in MLA decode, whose two CTAs exchange partial scores
# as fp16; its tests add that rounding's bound per row (assert_lse's `extra`).
F32_ATOL = 1e-5
BF16_ATOL = 1.5e-2
BF16_RTOL = 1e-2
BF16_LSE_ATOL = 1e-3


def dev(t, device="cuda"):
    return t.to(device) if isinstance(t, torch.Tensor) else t


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_parity(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, what: str = "out"):
    g = f64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: {np.count_nonzero(~np.isfinite(g))} non-finite values"
    d = np.abs(g - ref)
    if dtype == torch.float32:
        assert d.max() <= F32_ATOL, f"{what}: max abs err {d.max():.3e} > {F32_ATOL}"
    else:
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
        bad = d > bound
        assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance, "
                               f"max abs {d.max():.3e}, worst at {np.unravel_index(np.argmax(d - bound), d.shape)}")
    return float(d.max())


def assert_lse(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, extra: np.ndarray = None):
    """lse against the oracle; `extra` (shaped like ref) adds a per-element bound for
    a rounding step that the kernel takes on purpose (the MLA score exchange)."""
    g = f64(got)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(g), fin), "lse: -inf pattern differs"
    assert (g[~fin] == ref[~fin]).all()
    tol = np.full(ref.shape, F32_ATOL if dtype == torch.float32 else BF16_LSE_ATOL)
    if extra is not None:
        tol = tol + extra
    if fin.any():
        d = np.zeros(ref.shape)
        d[fin] = np.abs(g[fin] - ref[fin])
        worst = np.unravel_index(np.argmax(d - tol), d.shape)
        assert (d <= tol).all(), f"lse: max abs err {d.max():.3e}; at {worst} {d[worst]:.3e} > {tol[worst]:.3e}"


def replace_blocks(k_cache, v_cache, block_table, seq_lens, seed):
    """The same logical K/V moved to other physical blocks (a random permutation of the pool)."""
    nb = k_cache.shape[0]
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(nb).astype(np.int64))
    k2 = torch.empty_like(k_cache)
    v2 = torch.empty_like(v_cache)
    k2[perm] = k_cache
    v2[perm] = v_cache
    bt = block_table.clone().to(torch.int64)
    used = bt >= 0
    bt[used] = perm[bt[used]]
    return k2, v2, bt.to(torch.int32)
