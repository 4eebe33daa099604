"""Decode with the library's own choice of decomposition (pf_paged_attention_decode_auto)."""
import numpy as np
import pytest

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def test_plan_single_pass_for_many_items_and_split_for_a_long_few(pf):
    assert pf.decode_auto_plan(256, 32, 8, 128, 8192)[0] == 0          # 2048 items fill the GPU
    P, ws = pf.decode_auto_plan(4, 32, 8, 128, 131072)                   # 32 items, one very long
    assert P >= 256 and P & (P - 1) == 0 and ws == pf.partition_workspace_layout(4, 32, 128, 131072, P)[0]
    assert pf.decode_auto_plan(4, 32, 8, 128, 900)[0] == 0               # short contexts: one pass


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
