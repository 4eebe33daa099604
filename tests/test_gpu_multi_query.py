"""Multi-token paged query (pf_paged_attention_multi_query, which picks its kernel by row count,
and pf_paged_attention_multi_query_tcgen05) on the GPU against the oracle.

The last q_len tokens of every sequence are the new ones (already in the cache);
row (j, h) attends causally to the tokens t <= L - q_len + j."""
import numpy as np
import pytest
import torch

from tests.helpers import check_close, to_device
from workloads import BF16_NAN, make_workload, multi_query

pytestmark = pytest.mark.gpu


def run_multi(pf, d, q, kernel="auto"):
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    out = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                         kernel=kernel)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


CASES = [
    (32, 8, 128, 16, 1), (32, 8, 128, 16, 2), (32, 8, 128, 16, 4),    # Llama-3-8B heads, draft of 1-4 tokens
    (8, 8, 128, 16, 4), (8, 8, 128, 32, 16),                           # MHA, up to 16 new tokens
    (32, 4, 64, 16, 2), (4, 2, 64, 32, 8),                             # D=64 (g=8 q=2, g=2 q=8)
    (32, 8, 128, 16, 8), (32, 8, 128, 16, 16), (16, 8, 128, 32, 12),   # 32, 64 and 24 rows per kv head
    (32, 4, 64, 16, 6), (8, 8, 128, 16, 40), (4, 4, 64, 32, 64),       # 48 rows at D=64; MHA chunks of 40, 64
    (32, 8, 128, 16, 5), (16, 16, 128, 16, 3), (32, 8, 128, 48, 13),   # 20, 3 and 52 rows; a 48-token block
    (16, 4, 64, 16, 6), (8, 8, 64, 32, 20),                            # 24 and 20 rows at D=64 (two groups)
]
# the tcgen05 form is D = 128 only
KERNEL_CASES = [c + ("auto",) for c in CASES] + [c + ("tcgen05",) for c in CASES if c[2] == 128]


@pytest.mark.parametrize("Hq,Hkv,D,bs,Q,kernel", KERNEL_CASES)
def test_multi_query_matches_oracle(pf, oracle_lib, Hq, Hkv, D, bs, Q, kernel):
    lengths = [1, 3, 16, 17, 31, 64, 200, 513]
    wl = make_workload("mq", len(lengths), Hq, Hkv, D, bs, lengths, seed=Hq + D + bs + Q, pool_scale=2)
    q = multi_query(wl, Q)
    got = run_multi(pf, to_device(wl), q, kernel)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_multi_query_single_token_matches_decode(pf):
    wl = make_workload("mq1", 16, 32, 8, 128, 16, ("uniform", 1, 700), seed=101)
    d = to_device(wl)
    got = run_multi(pf, d, wl.q[:, None])[:, 0]
    dec = pf.paged_attention_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    check_close(got, dec.cpu().numpy(), abs_tol=2e-5, rel_tol=1e-4)


@pytest.mark.parametrize("kernel", ["auto", "tcgen05"])
def test_multi_query_llama3_shaped_batch(pf, oracle_lib, kernel):
    """64 sequences, 32 q / 8 kv heads, 4 draft tokens: every row against the oracle."""
    wl = make_workload("mq64", 64, 32, 8, 128, 16, ("uniform", 1024, 4096), seed=102)
    q = multi_query(wl, 4)
    got = run_multi(pf, to_device(wl), q, kernel)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


@pytest.mark.parametrize("kernel", ["auto", "tcgen05"])
def test_multi_query_wide_llama3_shaped_batch(pf, oracle_lib, kernel):
    """64 sequences, 32 q / 8 kv heads, 16 draft tokens (64 rows per kv head): every row."""
    wl = make_workload("mq64w", 64, 32, 8, 128, 16, ("uniform", 1024, 4096), seed=104)
    q = multi_query(wl, 16)
    got = run_multi(pf, to_device(wl), q, kernel)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


@pytest.mark.parametrize("kernel", ["auto", "tcgen05"])
def test_multi_query_wide_bad_block_and_length(pf, oracle_lib, kernel):
    """32 rows per kv head meet a table entry outside the pool and a length beyond the table:
    those sequences' rows are NaN, the others match the oracle, and the word is set."""
    wl = make_workload("mqbad", 4, 32, 8, 128, 16, [100, 70, 300, 33], seed=105, pool_scale=2)
    q = multi_query(wl, 8)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    d = to_device(wl)
    d["block_tables"][1, 2] = wl.num_blocks + 3
    d["context_lens"][2] = wl.block_tables.shape[1] * wl.block_size + 1
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    got = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], kernel=kernel).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    check_close(got[[0, 3]], ref[[0, 3]])


@pytest.mark.parametrize("q_len,kernel", [(4, "auto"), (8, "auto"), (16, "auto")])
def test_multi_query_llama3_full_size(pf, oracle_lib, config_workload, q_len, kernel):
    """The launches the bench times: all 256 Llama-3-shaped sequences (4.8 GB of K/V) with 4, 8
    and 16 draft tokens (16, 32 and 64 query rows per kv head: the three kernels the default
    entry picks), every row against the oracle."""
    wl = config_workload(4)
    q = multi_query(wl, q_len)
    got = run_multi(pf, to_device(wl), q, kernel)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["auto", "tcgen05"])
def test_multi_query_poisoned_new_token(pf, kernel):
    """A NaN key at the third new token of one sequence reaches exactly the rows whose causal
    window holds it: new tokens 2 .. q_len-1 of that kv head's query heads (the masked scores of
    the others are replaced, not multiplied).  A NaN value there reaches those rows too; the
    masked rows of the same kv head may see it through the 0 * NaN of the tensor-core P.V
    product, and nothing else may."""
    Q = 8
    wl = make_workload("mqnan", 3, 32, 8, 128, 16, [70, 130, 45], seed=107, pool_scale=2)
    q = multi_query(wl, Q)
    got = run_multi(pf, to_device(wl), q, kernel)
    assert np.isfinite(got).all()
    s, kv = 1, 3
    t = int(wl.context_lens[s]) - Q + 2
    blk, off = wl.block_tables[s, t // wl.block_size], t % wl.block_size
    expect = np.zeros(got.shape[:3], dtype=bool)
    expect[s, 2:, 4 * kv:4 * kv + 4] = True
    group = np.zeros_like(expect)
    group[s, :, 4 * kv:4 * kv + 4] = True
    for cache, exact in ((wl.k_cache, True), (wl.v_cache, False)):
        saved = cache[blk, kv, off].copy()
        cache[blk, kv, off, :] = BF16_NAN
        bad = np.isnan(run_multi(pf, to_device(wl), q, kernel)).any(axis=3)
        cache[blk, kv, off] = saved
        if exact:
            assert np.array_equal(bad, expect)
        else:
            assert bad[expect].all() and not bad[~group].any()


def test_multi_query_tcgen05_agrees_with_mma_sync(pf):
    """The tcgen05 kernel and the mma.sync kernels the default entry runs up to 32 rows per kv head
    agree to fp32 rounding at every such row count."""
    wl = make_workload("mqagree", 8, 32, 8, 128, 16, ("uniform", 1, 900), seed=108, pool_scale=2)
    d = to_device(wl)
    for Q in (1, 3, 4, 5, 8):
        q = multi_query(wl, Q)
        a, b = run_multi(pf, d, q, "auto"), run_multi(pf, d, q, "tcgen05")
        assert np.abs(a - b).max() <= 2e-5, Q


def test_multi_query_default_runs_tcgen05_past_32_rows(pf):
    """At head_dim 128 the default entry serves 33 to 64 rows per kv head with the tcgen05 kernel:
    its outputs are those of the explicit entry, bit for bit."""
    wl = make_workload("mqdisp", 8, 32, 8, 128, 16, ("uniform", 1, 900), seed=111, pool_scale=2)
    d = to_device(wl)
    for Q in (9, 12, 16):
        q = multi_query(wl, Q)
        assert np.array_equal(run_multi(pf, d, q, "auto"), run_multi(pf, d, q, "tcgen05")), Q


def test_multi_query_tcgen05_is_d128_only(pf):
    wl = make_workload("mqd64", 2, 8, 2, 64, 16, [40, 50], seed=109)
    d = to_device(wl)
    q = torch.zeros((2, 4, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pf.PFError) as e:
        pf.paged_attention_multi_query(q, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                       kernel="tcgen05")
    assert e.value.status == pf.PF_ERR_UNSUPPORTED


def test_multi_query_two_groups_repeated(pf):
    """32 query rows per kv head: two consumer groups take alternate stages of a 3-deep ring.
    200 launches back to back give bit-identical outputs and leave the error word clear (a group
    that waited on the wrong phase of a stage would read it early or stall)."""
    wl = make_workload("mqrep", 64, 32, 8, 128, 16, ("uniform", 256, 2048), seed=110)
    d = to_device(wl)
    qt = torch.from_numpy(np.ascontiguousarray(multi_query(wl, 8)).view(np.int16)).view(torch.bfloat16).cuda()
    args = (qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    first = pf.paged_attention_multi_query(*args)
    outs = [pf.paged_attention_multi_query(*args) for _ in range(200)]
    assert pf.get_device_error() == pf.PF_OK
    assert all(torch.equal(o, first) for o in outs)


def test_multi_query_tcgen05_repeated(pf):
    """64 rows per kv head through the tcgen05 kernel (the default entry's choice there): 100
    launches back to back give bit-identical outputs and leave the error word clear (a role that
    read a stage, a score buffer or P^T out of turn would change a result or stall)."""
    wl = make_workload("mqrep_tc", 64, 32, 8, 128, 16, ("uniform", 1, 3000), seed=112)
    d = to_device(wl)
    qt = torch.from_numpy(np.ascontiguousarray(multi_query(wl, 16)).view(np.int16)).view(torch.bfloat16).cuda()
    args = (qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    first = pf.paged_attention_multi_query(*args)
    outs = [pf.paged_attention_multi_query(*args) for _ in range(100)]
    assert pf.get_device_error() == pf.PF_OK
    assert all(torch.equal(o, first) for o in outs)
