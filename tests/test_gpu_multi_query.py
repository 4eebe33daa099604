"""Multi-token paged query (pf_paged_attention_multi_query) on the GPU against the oracle.

The last q_len tokens of every sequence are the new ones (already in the cache);
row (j, h) attends causally to the tokens t <= L - q_len + j."""
import numpy as np
import pytest
import torch

from tests.helpers import check_close, to_device
from workloads import make_workload, multi_query

pytestmark = pytest.mark.gpu


def run_multi(pf, d, q):
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    out = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


@pytest.mark.parametrize("Hq,Hkv,D,bs,Q", [
    (32, 8, 128, 16, 1), (32, 8, 128, 16, 2), (32, 8, 128, 16, 4),    # Llama-3-8B heads, draft of 1-4 tokens
    (8, 8, 128, 16, 4), (8, 8, 128, 32, 16),                           # MHA, up to 16 new tokens
    (32, 4, 64, 16, 2), (4, 2, 64, 32, 8),                             # D=64 (g=8 q=2, g=2 q=8)
    (32, 8, 128, 16, 8), (32, 8, 128, 16, 16), (16, 8, 128, 32, 12),   # 32, 64 and 24 rows per kv head
    (32, 4, 64, 16, 6), (8, 8, 128, 16, 40), (4, 4, 64, 32, 64),       # 48 rows at D=64; MHA chunks of 40, 64
])
def test_multi_query_matches_oracle(pf, oracle_lib, Hq, Hkv, D, bs, Q):
    lengths = [1, 3, 16, 17, 31, 64, 200, 513]
    wl = make_workload("mq", len(lengths), Hq, Hkv, D, bs, lengths, seed=Hq + D + bs + Q, pool_scale=2)
    q = multi_query(wl, Q)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_multi_query_single_token_matches_decode(pf):
    wl = make_workload("mq1", 16, 32, 8, 128, 16, ("uniform", 1, 700), seed=101)
    d = to_device(wl)
    got = run_multi(pf, d, wl.q[:, None])[:, 0]
    dec = pf.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    check_close(got, dec.cpu().numpy(), abs_tol=2e-5, rel_tol=1e-4)


def test_multi_query_llama3_shaped_batch(pf, oracle_lib):
    """64 sequences, 32 q / 8 kv heads, 4 draft tokens: every row against the oracle."""
    wl = make_workload("mq64", 64, 32, 8, 128, 16, ("uniform", 1024, 4096), seed=102)
    q = multi_query(wl, 4)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_multi_query_wide_llama3_shaped_batch(pf, oracle_lib):
    """64 sequences, 32 q / 8 kv heads, 16 draft tokens (64 rows per kv head): every row."""
    wl = make_workload("mq64w", 64, 32, 8, 128, 16, ("uniform", 1024, 4096), seed=104)
    q = multi_query(wl, 16)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_multi_query_wide_bad_block_and_length(pf, oracle_lib):
    """The 32-row kernel meets a table entry outside the pool and a length beyond the table:
    those sequences' rows are NaN, the others match the oracle, and the word is set."""
    wl = make_workload("mqbad", 4, 32, 8, 128, 16, [100, 70, 300, 33], seed=105, pool_scale=2)
    q = multi_query(wl, 8)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    d = to_device(wl)
    d["block_tables"][1, 2] = wl.num_blocks + 3
    d["context_lens"][2] = wl.block_tables.shape[1] * wl.block_size + 1
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    got = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"]).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    check_close(got[[0, 3]], ref[[0, 3]])


def test_multi_query_rows_beyond_sixty_four_are_unsupported(pf):
    wl = make_workload("mqx", 2, 32, 8, 128, 16, [40, 50], seed=103)
    d = to_device(wl)
    q = torch.zeros((2, 17, 32, 128), dtype=torch.bfloat16, device="cuda")     # g=4 x 17 = 68 rows
    with pytest.raises(pf.PFError) as e:
        pf.paged_attention_multi_query(q, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    assert e.value.status == pf.PF_ERR_UNSUPPORTED


@pytest.mark.parametrize("q_len", [4, 16])
def test_multi_query_llama3_full_size(pf, oracle_lib, config_workload, q_len):
    """The launches the bench times: all 256 Llama-3-shaped sequences (4.8 GB of K/V) with 4
    and with 16 draft tokens (16 and 64 query rows per kv head), every row against the oracle."""
    wl = config_workload(4)
    q = multi_query(wl, q_len)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    torch.cuda.empty_cache()
