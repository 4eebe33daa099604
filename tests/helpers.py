"""Test-side helpers: gathers and scatters written with numpy indexing.

They are deliberately a second, independent route to the same quantities
(the oracle loops token by token in C); nothing here is used by the product.
"""
from __future__ import annotations

import numpy as np

from workloads import bf16_bits_to_f32


def gather_kv(wl, i, k_cache=None, v_cache=None):
    """Contiguous K, V of sequence i as float64 arrays [L, Hkv, D] (numpy fancy indexing)."""
    kc = wl.k_cache if k_cache is None else k_cache
    vc = wl.v_cache if v_cache is None else v_cache
    L = int(wl.context_lens[i])
    t = np.arange(L)
    blk = wl.block_tables[i, t // wl.block_size]
    off = t % wl.block_size
    K = bf16_bits_to_f32(kc[blk, :, off, :]).astype(np.float64)
    V = bf16_bits_to_f32(vc[blk, :, off, :]).astype(np.float64)
    return K, V


def q_f64(wl):
    return bf16_bits_to_f32(wl.q).astype(np.float64)


def numpy_scatter(wl):
    """Cache state after the append, by numpy fancy indexing."""
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    s = wl.slot_mapping
    ok = s >= 0
    blk, off = s[ok] // wl.block_size, s[ok] % wl.block_size
    kc[blk, :, off, :] = wl.new_k[ok]
    vc[blk, :, off, :] = wl.new_v[ok]
    return kc, vc


def check_close(got, ref, abs_tol=2e-3, rel_tol=1e-2, rel_floor=0.2):
    """Attention tolerance: max |d| <= abs_tol, and |d|/|ref| <= rel_tol where |ref| >= rel_floor.

    Returns (max_abs, max_rel) and raises AssertionError with both when either bound fails.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    d = np.abs(got - ref)
    max_abs = float(d.max()) if d.size else 0.0
    big = np.abs(ref) >= rel_floor
    max_rel = float((d[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    assert max_abs <= abs_tol and max_rel <= rel_tol, f"max_abs={max_abs:.3e} max_rel={max_rel:.3e}"
    return max_abs, max_rel
