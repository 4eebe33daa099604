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
    """64 sequences, 32 q / 8 kv heads, 4 draft tokens: sampled rows against the oracle."""
    wl = make_workload("mq64", 64, 32, 8, 128, 16, ("uniform", 1024, 4096), seed=102)
    q = multi_query(wl, 4)
    got = run_multi(pf, to_device(wl), q)
    assert np.all(np.isfinite(got))
    idx = np.random.default_rng(0).choice(64, size=6, replace=False)
    sub = dict(q=q[idx], block_tables=wl.block_tables[idx], context_lens=wl.context_lens[idx])
    ref = oracle_lib.paged_attention_multi(sub["q"], wl.k_cache, wl.v_cache, sub["block_tables"], sub["context_lens"],
                                           wl.scale)
    check_close(got[idx], ref)


def test_multi_query_rows_beyond_sixteen_are_unsupported(pf):
    wl = make_workload("mqx", 2, 32, 8, 128, 16, [40, 50], seed=103)
    d = to_device(wl)
    q = torch.zeros((2, 5, 32, 128), dtype=torch.bfloat16, device="cuda")      # g=4 x 5 = 20 rows
    with pytest.raises(pf.PFError) as e:
        pf.paged_attention_multi_query(q, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    assert e.value.status == pf.PF_ERR_UNSUPPORTED
