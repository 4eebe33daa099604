"""Batches past the in-CTA sorting limits: above 512 sequences the decode and the fused
append+decode map CTAs to items in natural order, and above 1,024 the partition pass
runs one CTA per (sequence, partition, kv head) instead of the persistent kernel."""
import numpy as np
import pytest

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def test_decode_above_512_sequences(pf, oracle_lib):
    wl = make_workload("big", 700, 8, 2, 64, 16, ("uniform", 0, 150), seed=81)
    got = pf.paged_attention_decode(*attn_args(to_device(wl))).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_fused_append_decode_above_512_sequences(pf, oracle_lib):
    wl = make_workload("bigapp", 600, 4, 4, 128, 16, ("uniform", 1, 120), seed=82, append=True,
                       num_skip_slots=20)
    d = to_device(wl)
    got = pf.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"],
                                           d["v_cache"], d["block_tables"], d["context_lens"]).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    kc, vc, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                             wl.block_size)
    ref = oracle_lib.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_split_above_1024_sequences(pf, oracle_lib):
    wl = make_workload("bigsplit", 1100, 8, 2, 64, 16, ("uniform", 0, 300), seed=83)
    d = to_device(wl)
    P, mx = 64, wl.max_context_len
    ws = pf.alloc_workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, mx, P, "cuda")
    pf.paged_attention_decode_partition(*attn_args(d), P, mx, ws)
    got = pf.paged_attention_merge(ws, d["context_lens"], wl.num_q_heads, wl.head_dim, P, mx).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    assert not got[wl.context_lens == 0].any()


@pytest.mark.parametrize("q_len", [2, 8])
def test_multi_query_above_512_sequences(pf, oracle_lib, q_len):
    """Past 512 sequences the multi-token kernels (16-row and wide) take natural order."""
    import torch
    from workloads import multi_query
    wl = make_workload("bigmq", 600, 16, 4, 64, 16, ("uniform", 1, 90), seed=84 + q_len)
    q = multi_query(wl, q_len)
    d = to_device(wl)
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    got = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"]).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
