"""Single-pass paged decode attention on the GPU against the fp64 oracle.

Tolerance (fp32 accumulation of bf16 inputs against fp64): max |d| <= 2e-3 and
|d|/|ref| <= 1e-2 on elements with |ref| >= 0.2.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, gather_kv, to_device
from workloads import BF16_NAN, make_workload

pytestmark = pytest.mark.gpu


def decode(pf, d, **kw):
    out = pf.paged_attention_decode(*attn_args(d), **kw)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


def oracle_out(orc, wl, k_cache=None, v_cache=None, threads=0):
    return orc.paged_attention(wl.q, wl.k_cache if k_cache is None else k_cache,
                               wl.v_cache if v_cache is None else v_cache, wl.block_tables, wl.context_lens,
                               wl.scale, threads=threads)


@pytest.mark.parametrize("index", [1, 2])
def test_named_workloads_full(pf, oracle_lib, config_workload, index):
    wl = config_workload(index)
    got = decode(pf, to_device(wl))
    check_close(got, oracle_out(oracle_lib, wl))


def test_cont_batch_append_then_decode(pf, oracle_lib, config_workload):
    """The continuous-batch step: append one token per sequence (8 padded), then attend."""
    wl = config_workload(3)
    d = to_device(wl)
    pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    got = decode(pf, d)
    kc, vc, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                             wl.block_size)
    check_close(got, oracle_out(oracle_lib, wl, kc, vc))


def test_llama3_8b_full_size(pf, oracle_lib, config_workload):
    """256 sequences, 4.8 GB of KV, the launch the bench times: every output row against the
    oracle (about a second of the host's cores)."""
    wl = config_workload(4)
    got = decode(pf, to_device(wl))
    check_close(got, oracle_out(oracle_lib, wl))
    torch.cuda.empty_cache()


def test_long_context_single_pass(pf, oracle_lib, config_workload):
    """The 131072-token sequence through the single-pass kernel (one CTA per kv head)."""
    wl = config_workload(5)
    got = decode(pf, to_device(wl))
    check_close(got, oracle_out(oracle_lib, wl))


EDGE_LENGTHS = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_edge_lengths_all_variants(pf, oracle_lib, D, bs, g):
    Hkv = 2
    wl = make_workload("edge", len(EDGE_LENGTHS), Hkv * g, Hkv, D, bs, EDGE_LENGTHS, seed=D * 100 + bs * 10 + g,
                       pool_scale=2)
    check_close(decode(pf, to_device(wl)), oracle_out(oracle_lib, wl))


def test_single_sequence_and_zero_length(pf, oracle_lib):
    wl = make_workload("one", 1, 8, 2, 128, 16, [300], seed=31)
    check_close(decode(pf, to_device(wl)), oracle_out(oracle_lib, wl))
    wl = make_workload("zero", 3, 4, 4, 64, 16, [0, 5, 0], seed=32)
    got = decode(pf, to_device(wl))
    assert np.array_equal(got[0], np.zeros_like(got[0])) and np.array_equal(got[2], np.zeros_like(got[2]))
    check_close(got, oracle_out(oracle_lib, wl))


def test_length_one_returns_v_exactly(pf):
    wl = make_workload("l1", 5, 16, 4, 128, 16, [1] * 5, seed=33, pool_scale=3)
    got = decode(pf, to_device(wl))
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        for h in range(wl.num_q_heads):
            assert np.array_equal(got[i, h], V[0, h // wl.group].astype(np.float32))


def test_block_permutation_gives_bit_identical_output(pf, config_workload):
    wl = config_workload(2)
    base = decode(pf, to_device(wl))
    perm = np.random.default_rng(7).permutation(wl.num_blocks)
    kc, vc = np.empty_like(wl.k_cache), np.empty_like(wl.v_cache)
    kc[perm], vc[perm] = wl.k_cache, wl.v_cache
    tables = wl.block_tables.copy()
    nblk = (wl.context_lens + wl.block_size - 1) // wl.block_size
    for i in range(wl.num_seqs):
        tables[i, :nblk[i]] = perm[tables[i, :nblk[i]]]
    wl2 = dataclasses.replace(wl, k_cache=kc, v_cache=vc, block_tables=tables)
    assert np.array_equal(decode(pf, to_device(wl2)), base)


def test_deterministic(pf, config_workload):
    d = to_device(config_workload(3))
    pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    a = decode(pf, d)
    b = decode(pf, d)
    assert np.all(np.isfinite(a)) and np.array_equal(a, b)


def test_poison_is_never_read(pf, oracle_lib):
    """Tails, unused blocks and table entries past the end are poison; a valid row must stay finite,
    and poisoning a *valid* token must reach exactly the rows that read it."""
    wl = make_workload("poison", 4, 8, 2, 128, 16, [3, 16, 17, 40], seed=34, pool_scale=3)
    d = to_device(wl)
    got = decode(pf, d)
    assert np.all(np.isfinite(got))
    b = wl.block_tables[3, 1]
    wl.v_cache[b, 1, 4, :] = BF16_NAN                        # seq 3, kv head 1, token 20
    got2 = decode(pf, to_device(wl))
    bad = ~np.isfinite(got2).all(axis=2)
    expect = np.zeros_like(bad)
    expect[3, 4:8] = True
    assert np.array_equal(bad, expect)
    b = wl.block_tables[1, 0]
    wl.k_cache[b, 0, 7, :] = BF16_NAN                        # seq 1, kv head 0, token 7: a NaN score
    got3 = decode(pf, to_device(wl))
    bad = ~np.isfinite(got3).all(axis=2)
    expect[1, 0:4] = True
    assert np.array_equal(bad, expect)
    assert np.isnan(got3[1, 0:4]).all()                       # NaN, not a silent zero


def test_nan_key_in_the_decode_without_its_append(pf, oracle_lib, config_workload):
    """The continuous-batch cache before its append holds NaN in every slot about to be
    filled (position L-1 of 56 sequences): those rows are NaN, as in the oracle."""
    wl = config_workload(3)
    got = decode(pf, to_device(wl))
    ref = oracle_out(oracle_lib, wl)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    rows = ~np.isnan(ref).any(axis=(1, 2))
    assert rows.sum() == 8                                     # the 8 sequences that append nothing
    check_close(got[rows], ref[rows])


def test_scale_argument(pf, oracle_lib):
    wl = make_workload("scale", 3, 8, 8, 64, 32, [50, 64, 70], seed=35)
    d = to_device(wl)
    for scale in (0.0, 0.05, 0.4):
        got = decode(pf, d, scale=scale)
        ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, scale)
        check_close(got, ref)


def test_other_block_sizes(pf, oracle_lib):
    """Any multiple of 16 works (tiles of 16 tokens); 64 and 48 are beyond the named workloads."""
    for bs in (48, 64):
        wl = make_workload("bs", 3, 8, 2, 128, bs, [47, 100, 130], seed=bs)
        check_close(decode(pf, to_device(wl)), oracle_out(oracle_lib, wl))
