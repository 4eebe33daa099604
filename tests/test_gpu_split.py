"""Split over context partitions (partition pass + log-sum-exp merge) on the GPU."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def split(pf, d, wl, P, max_ctx=None):
    max_ctx = wl.max_context_len if max_ctx is None else max_ctx
    ws = pf.alloc_workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, max_ctx, P, "cuda")
    pf.paged_attention_decode_partition(*attn_args(d), P, max_ctx, ws)
    out = pf.paged_attention_merge(ws, d["context_lens"], wl.num_q_heads, wl.head_dim, P, max_ctx)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy(), ws, max_ctx


def test_long_skew_full(pf, oracle_lib, config_workload):
    """131072 + 3 x 512 tokens, 512-token partitions: every output row against the oracle."""
    wl = config_workload(5)
    got, _, _ = split(pf, to_device(wl), wl, wl.partition_size)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    torch.cuda.empty_cache()


def test_partials_match_oracle_partials(pf, oracle_lib):
    wl = make_workload("parts", 3, 8, 2, 128, 16, [1000, 512, 33], seed=41)
    P = 256
    d = to_device(wl)
    _, ws, max_ctx = split(pf, d, wl, P)
    o, m, l = (t.cpu().numpy() for t in pf.workspace_views(ws, wl.num_seqs, wl.num_q_heads, wl.head_dim,
                                                            max_ctx, P))
    ro, rm, rl = oracle_lib.partition(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, P)
    for i in range(wl.num_seqs):
        npart = -(-int(wl.context_lens[i]) // P)
        check_close(o[i, :, :npart], ro[i, :, :npart])
        np.testing.assert_allclose(m[i, :, :npart], rm[i, :, :npart], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(l[i, :, :npart], rl[i, :, :npart], rtol=1e-4)


@pytest.mark.parametrize("P", [16, 64, 512, 4096])
@pytest.mark.parametrize("D,g,bs", [(128, 4, 32), (64, 8, 16), (128, 1, 16)])
def test_split_equals_unsplit(pf, oracle_lib, P, D, g, bs):
    wl = make_workload("split", 4, 2 * g, 2, D, bs, [1, 300, 1025, 2000], seed=P + D + g + bs)
    d = to_device(wl)
    got, _, _ = split(pf, d, wl, P)
    one = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    check_close(got, one, abs_tol=1e-5, rel_tol=1e-4)


def test_max_context_len_above_lengths_and_empty_sequences(pf, oracle_lib):
    wl = make_workload("ws", 4, 4, 4, 64, 16, [0, 40, 700, 0], seed=42)
    got, _, _ = split(pf, to_device(wl), wl, 128, max_ctx=2048)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    assert not got[0].any() and not got[3].any()
    check_close(got, ref)


def test_workspace_too_small_is_rejected(pf):
    wl = make_workload("ws", 2, 4, 4, 64, 16, [40, 70], seed=43)
    d = to_device(wl)
    total = pf.partition_workspace_layout(2, 4, 64, 70, 32)[0]
    ws = torch.empty(total - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pf.PFError) as e:
        pf.paged_attention_decode_partition(*attn_args(d), 32, 70, ws)
    assert e.value.status == pf.PF_ERR_INVALID_ARG


@pytest.mark.parametrize("D", [64, 128])
def test_merge_many_partitions(pf, oracle_lib, D):
    """More partitions per row than one batch of the merge's loads (313 at P=16): the
    statistics and the weighted sums run over several batches with a ragged last one."""
    wl = make_workload("manyparts", 4, 8, 2, D, 16, [5000, 4097, 16, 1], seed=44 + D)
    d = to_device(wl)
    got, _, _ = split(pf, d, wl, 16)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
