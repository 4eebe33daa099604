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


def to_device(wl, device="cuda"):
    """The workload's arrays as CUDA tensors (bf16 tensors carry the same bits)."""
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    d = dict(q=bf(wl.q), k_cache=bf(wl.k_cache), v_cache=bf(wl.v_cache),
             block_tables=torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(device),
             context_lens=torch.from_numpy(np.ascontiguousarray(wl.context_lens)).to(device))
    if wl.slot_mapping is not None:
        d.update(new_k=bf(wl.new_k), new_v=bf(wl.new_v),
                 slot_mapping=torch.from_numpy(np.ascontiguousarray(wl.slot_mapping)).to(device))
    return d


def bits(t):
    """bf16 CUDA tensor -> uint16 numpy array of its bits."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def attn_args(d):
    return d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"]
