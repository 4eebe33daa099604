"""Decode with the library's own choice of decomposition (pf_paged_attention_decode_auto)."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def test_plan_single_pass_for_many_items_and_split_for_a_long_few(pf):
    assert pf.decode_auto_plan(256, 32, 8, 128, 8192)[0] == 0          # 2048 items fill the GPU
    P, ws = pf.decode_auto_plan(4, 32, 8, 128, 131072)                   # 32 items, one very long
    assert P >= 256 and P & (P - 1) == 0 and ws == pf.partition_workspace_layout(4, 32, 128, 131072, P)[0]
    assert pf.decode_auto_plan(200, 32, 8, 128, 900)[0] == 0             # many items, short contexts: one pass
    # few items, contexts a cluster of 8 covers in chunks of <= 1024 tokens: the cluster split
    # (a chunk size, no workspace)
    P, ws = pf.decode_auto_plan(4, 32, 8, 128, 900)
    assert ws == 0 and P == 128                                          # 57 tiles over 8 CTAs
    P, ws = pf.decode_auto_plan(4, 4, 2, 64, 64)                         # the tiny workload: 4 CTAs of 16 tokens
    assert ws == 0 and P == 16


def test_auto_long_skew_uses_split_and_matches_oracle(pf, oracle_lib, config_workload):
    wl = config_workload(5)
    P, _ = pf.decode_auto_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.max_context_len)
    assert P > 0
    d = to_device(wl)
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=wl.max_context_len).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_auto_single_pass_equals_decode(pf):
    wl = make_workload("auto", 40, 16, 4, 128, 16, ("uniform", 10, 900), seed=91)
    d = to_device(wl)
    assert pf.decode_auto_plan(40, 16, 4, 128, wl.max_context_len)[0] == 0
    a = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=wl.max_context_len).cpu().numpy()
    b = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    assert np.array_equal(a, b)


def _cluster_plan(pf, wl):
    P, ws = pf.decode_auto_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.max_context_len)
    return P, ws


@pytest.mark.parametrize("index", [1, 2])
def test_auto_cluster_split_on_the_small_workloads(pf, oracle_lib, config_workload, index):
    """The tiny and TinyLlama-shaped workloads have few (sequence, kv head) items: the auto decode
    runs the cluster split (no workspace) and matches the oracle."""
    wl = config_workload(index)
    P, ws = _cluster_plan(pf, wl)
    assert P > 0 and ws == 0
    d = to_device(wl)
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=wl.max_context_len).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


# (Hq, Hkv, D, bs, lengths): every group, both head dims, block sizes 16/32/48, empty and
# one-token sequences, lengths on and off chunk boundaries, chunks past a sequence's end
CLUSTER_CASES = [
    (8, 8, 128, 16, [0, 1, 16, 17, 300, 1000]),
    (16, 8, 128, 32, [5, 64, 65, 999, 1024, 2]),
    (32, 8, 64, 16, [129, 0, 700, 33]),
    (32, 4, 64, 48, [1, 2000, 47, 48, 49]),
    (64, 8, 128, 16, [4000, 12, 3000]),
    (4, 2, 64, 16, [1, 17, 33, 64]),
]


@pytest.mark.parametrize("Hq,Hkv,D,bs,lengths", CLUSTER_CASES)
def test_auto_cluster_split_matches_oracle(pf, oracle_lib, Hq, Hkv, D, bs, lengths):
    wl = make_workload("clu", len(lengths), Hq, Hkv, D, bs, lengths, seed=Hq + D + bs + len(lengths), pool_scale=2)
    mx = max(wl.max_context_len, 32)
    P, ws = pf.decode_auto_plan(wl.num_seqs, Hq, Hkv, D, mx)
    assert P > 0 and ws == 0
    d = to_device(wl)
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    for i, L in enumerate(lengths):
        if L == 0:
            assert not got[i].any()


def test_auto_cluster_split_bad_length_and_block(pf, oracle_lib):
    """A length beyond max_context_len and a table entry outside the pool: those sequences' rows
    are NaN, the others match the oracle, the error word says so; repeated calls are bit-identical."""
    wl = make_workload("clubad", 4, 16, 4, 128, 16, [300, 200, 500, 150], seed=93, pool_scale=2)
    mx = wl.max_context_len
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    d = to_device(wl)
    d["block_tables"][1, 3] = wl.num_blocks + 5
    d["context_lens"][2] = mx + 1
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx)
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    g = got.cpu().numpy()
    assert np.isnan(g[1]).all() and np.isnan(g[2]).all()
    check_close(g[[0, 3]], ref[[0, 3]])
    d["block_tables"][1, 3] = int(wl.block_tables[1, 3])
    d["context_lens"][2] = int(wl.context_lens[2])
    first = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx)
    outs = [pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx) for _ in range(50)]
    assert pf.get_device_error() == pf.PF_OK
    assert all(torch.equal(o, first) for o in outs)
    check_close(first.cpu().numpy(), ref)


def _split_plan(pf, wl, mx):
    P, ws = pf.decode_auto_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, mx)
    assert P > 0 and ws > 0, "the workspace split"
    return P, ws


# Batches the auto decode splits over context partitions (S, Hq, Hkv, D, bs, lengths,
# max_context_len): every group, both head dims, block sizes 16/32/48; empty and one-token
# rows, lengths on and off 16-token tiles and partition boundaries, one row much longer
# than the rest, and a batch far shorter than max_context_len.
SPLIT_CASES = [
    (20, 32, 8, 128, 16, [0, 1, 15, 16, 17, 1025, 3000, 33, 2048, 0, 7, 900, 1600, 64, 65, 2, 1999, 480, 31, 3000], 3000),
    (12, 64, 8, 64, 32, [5000, 1, 4096, 33, 0, 2500, 32, 31, 4000, 1200, 64, 4999], 5000),
    (10, 16, 16, 128, 48, [1100, 47, 48, 49, 0, 2200, 3, 96, 1500, 700], 2200),
    (2, 8, 4, 128, 16, [20000, 3], 20000),
    (10, 16, 8, 128, 16, [1, 16, 17, 64, 0, 33, 48, 50, 2, 63], 2000),
    (12, 8, 8, 64, 16, [0] * 12, 2000),
]


@pytest.mark.parametrize("S,Hq,Hkv,D,bs,lengths,mx", SPLIT_CASES)
def test_auto_split_matches_oracle(pf, oracle_lib, S, Hq, Hkv, D, bs, lengths, mx):
    wl = make_workload("autosplit", S, Hq, Hkv, D, bs, lengths, seed=S + Hq + D + bs, pool_scale=2)
    _split_plan(pf, wl, mx)
    d = to_device(wl)
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    for i, L in enumerate(lengths):
        if L == 0:
            assert not got[i].any()


def test_auto_split_ignores_workspace_contents_and_repeats(pf, oracle_lib):
    """The workspace is scratch: NaN-filled or random bytes give the same bits; 30 repeats agree."""
    wl = make_workload("autows", 12, 32, 8, 128, 16, ("uniform", 1, 6000), seed=97, pool_scale=2)
    mx = 6000
    _, ws = _split_plan(pf, wl, mx)
    d = to_device(wl)
    w = torch.empty(ws, dtype=torch.uint8, device="cuda")
    w.view(torch.float32)[: ws // 4].fill_(float("nan"))
    first = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx, workspace=w)
    g = torch.Generator(device="cuda").manual_seed(5)
    w.copy_(torch.randint(0, 256, (ws,), dtype=torch.uint8, device="cuda", generator=g))
    second = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx, workspace=w)
    outs = [pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx, workspace=w) for _ in range(30)]
    assert pf.get_device_error() == pf.PF_OK
    assert torch.equal(first, second) and all(torch.equal(o, first) for o in outs)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(first.cpu().numpy(), ref)


def test_auto_split_bad_length_and_block(pf, oracle_lib):
    """A length beyond max_context_len and table entries outside the pool, in a long row and in
    a short one: those sequences' rows are NaN, the others match the oracle, the error word says so."""
    lengths = [30000, 500, 200, 40000, 300, 100, 800, 20]
    wl = make_workload("autobad", 8, 32, 8, 128, 16, lengths, seed=99, pool_scale=2)
    mx = 40000
    _split_plan(pf, wl, mx)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    d = to_device(wl)
    d["block_tables"][0, 1000] = wl.num_blocks + 5
    d["block_tables"][4, 2] = -1
    d["context_lens"][6] = mx + 1
    got = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx)
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    g = got.cpu().numpy()
    for i in (0, 4, 6):
        assert np.isnan(g[i]).all(), i
    keep = [1, 2, 3, 5, 7]
    check_close(g[keep], ref[keep])


def test_auto_split_equals_decode_within_rounding(pf):
    wl = make_workload("autoeq", 16, 32, 8, 128, 32, ("loguniform", 16, 16000), seed=101, pool_scale=2)
    mx = int(wl.max_context_len)
    _split_plan(pf, wl, mx)
    d = to_device(wl)
    a = pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx)
    b = pf.paged_attention_decode(*attn_args(d))
    assert pf.get_device_error() == pf.PF_OK
    torch.testing.assert_close(a, b, rtol=1e-4, atol=1e-5)
