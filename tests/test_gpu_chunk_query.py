"""Multi-token query past 64 rows per kv head -- prompt chunks -- on the GPU against the oracle.

pf_paged_attention_multi_query serves more than 64 query rows per kv head (g * q_len) with the
prompt-chunk kernel: one CTA per (sequence, kv head, 128-row tile), the query rows on the M
side of tcgen05.mma.  The last q_len tokens of every sequence are the chunk (already in the
cache); row (j, h) attends to the tokens t <= L - q_len + j, and rows whose position is
negative (L < q_len) are zero."""
import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import check_close, to_device
from workloads import BF16_NAN, make_workload, multi_query

pytestmark = pytest.mark.gpu

LENGTHS = [1, 3, 16, 17, 31, 64, 127, 128, 129, 200, 513, 1000]


def run_multi(pf, d, q, kernel="auto"):
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    out = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                         kernel=kernel)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


# (Hq, Hkv, D, bs, q_len): g in {1, 4} with q_len in {17, 32, 64, 128} where g * q_len > 64,
# other groups, head_dim 64, block sizes 16, 32 and 48 (not a power of two), and odd numbers
# of row tiles
CASES = [
    (32, 8, 128, 16, 17), (32, 8, 128, 16, 32), (32, 8, 128, 16, 64), (32, 8, 128, 16, 128),  # g = 4
    (8, 8, 128, 16, 128), (8, 8, 128, 32, 65), (4, 4, 128, 16, 200),                        # g = 1
    (16, 8, 128, 32, 40), (64, 8, 128, 16, 9), (32, 8, 128, 48, 33),                        # g = 2, 8; bs 48
    (32, 4, 64, 16, 16), (8, 2, 64, 32, 64), (8, 8, 64, 16, 130), (32, 8, 64, 16, 48),      # head_dim 64
    # an odd number of 128-row tiles (the last cluster pair has an empty second tile)
    (32, 8, 128, 16, 80), (8, 8, 128, 16, 300), (32, 8, 64, 32, 100),
]


@pytest.mark.parametrize("Hq,Hkv,D,bs,Q", CASES)
def test_chunk_query_matches_oracle(pf, oracle_lib, Hq, Hkv, D, bs, Q):
    wl = make_workload("cq", len(LENGTHS), Hq, Hkv, D, bs, LENGTHS, seed=Hq + D + bs + Q, pool_scale=2)
    q = multi_query(wl, Q)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    # positions before the sequence start give zero rows
    for i, L in enumerate(LENGTHS):
        if L < Q:
            assert not got[i, :Q - L].any()


@pytest.mark.parametrize("Q", [17, 64])
def test_chunk_query_tcgen05_entry_is_the_same_kernel(pf, Q):
    """Past 64 rows the explicit tcgen05 entry runs the same prompt-chunk kernel: bit for bit."""
    wl = make_workload("cqtc", 6, 32, 8, 128, 16, [40, 300, 1, 64, 900, 128], seed=120 + Q, pool_scale=2)
    d = to_device(wl)
    q = multi_query(wl, Q)
    assert np.array_equal(run_multi(pf, d, q, "auto"), run_multi(pf, d, q, "tcgen05"))


def test_chunk_query_llama3_full_size(pf, oracle_lib, config_workload):
    """The launch the bench times: all 256 Llama-3-shaped sequences (4.8 GB of K/V) with a
    64-token chunk each (256 query rows per kv head, two row tiles), every row against the oracle."""
    wl = config_workload(4)
    q = multi_query(wl, 64)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    torch.cuda.empty_cache()


def test_chunk_query_long_chunk_few_sequences(pf, oracle_lib):
    """A 512-token chunk at the end of 3 000- to 6 000-token contexts (2 048 rows per kv head:
    16 row tiles of one kv head read the same K/V tiles)."""
    wl = make_workload("cqlong", 3, 32, 8, 128, 16, [3000, 512, 6000], seed=125)
    q = multi_query(wl, 512)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_chunk_query_dominant_keys(pf, oracle_lib):
    """Keys scaled by 8 (outlier rows) make the softmax concentrated and move the reference maximum
    late in a sequence; the probabilities' hi + lo split keeps the result within tolerance."""
    wl = make_workload("cqout", 8, 32, 8, 128, 16, ("uniform", 100, 2000), seed=126, outlier_frac=0.02)
    q = multi_query(wl, 32)
    got = run_multi(pf, to_device(wl), q)
    ref = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)


def test_chunk_query_bad_block_and_length(pf, oracle_lib):
    """A table entry outside the pool and a length beyond the table: those sequences' rows are
    NaN, the others match the oracle, and the error word says so."""
    wl = make_workload("cqbad", 4, 32, 8, 128, 16, [300, 200, 500, 150], seed=127, pool_scale=2)
    q = multi_query(wl, 40)
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


def test_chunk_query_poisoned_chunk_token(pf):
    """A NaN key at the fifth token of one sequence's chunk reaches exactly the rows whose causal
    window holds it (new tokens 4 .. q_len-1 of that kv head's query heads); a NaN value there
    reaches those rows too, and may reach only the other rows of the same kv head (through
    0 * NaN in P.V)."""
    Q = 40
    wl = make_workload("cqnan", 3, 32, 8, 128, 16, [170, 230, 45], seed=128, pool_scale=2)
    q = multi_query(wl, Q)
    got = run_multi(pf, to_device(wl), q)
    assert np.isfinite(got).all()
    s, kv = 1, 5
    t = int(wl.context_lens[s]) - Q + 4
    blk, off = wl.block_tables[s, t // wl.block_size], t % wl.block_size
    expect = np.zeros(got.shape[:3], dtype=bool)
    expect[s, 4:, 4 * kv:4 * kv + 4] = True
    group = np.zeros_like(expect)
    group[s, :, 4 * kv:4 * kv + 4] = True
    for cache, exact in ((wl.k_cache, True), (wl.v_cache, False)):
        saved = cache[blk, kv, off].copy()
        cache[blk, kv, off, :] = BF16_NAN
        bad = np.isnan(run_multi(pf, to_device(wl), q)).any(axis=3)
        cache[blk, kv, off] = saved
        if exact:
            assert np.array_equal(bad, expect)
        else:
            assert bad[expect].all() and not bad[~group].any()


def test_chunk_query_repeated(pf):
    """100 launches back to back give bit-identical outputs and leave the error word clear (a role
    that read a stage, a score buffer or P out of turn would change a result or stall)."""
    wl = make_workload("cqrep", 32, 32, 8, 128, 16, ("uniform", 1, 3000), seed=129)
    d = to_device(wl)
    qt = torch.from_numpy(np.ascontiguousarray(multi_query(wl, 64)).view(np.int16)).view(torch.bfloat16).cuda()
    args = (qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    first = pf.paged_attention_multi_query(*args)
    outs = [pf.paged_attention_multi_query(*args) for _ in range(100)]
    assert pf.get_device_error() == pf.PF_OK
    assert all(torch.equal(o, first) for o in outs)


def test_chunk_query_rows_beyond_the_limit_are_unsupported(pf):
    """g * q_len above 65 536 rows per kv head is refused before anything is launched."""
    wl = make_workload("cqx", 2, 32, 8, 128, 16, [40, 50], seed=130)
    d = to_device(wl)
    q = torch.zeros((2, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((2, 1, 32, 128), dtype=torch.float32, device="cuda")
    f = pf.lib().pf_paged_attention_multi_query
    for q_len, want in ((16385, pf.PF_ERR_UNSUPPORTED), (0, pf.PF_ERR_INVALID_ARG)):   # 4 x 16 385 = 65 540 rows
        st = f(q.data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(), d["block_tables"].data_ptr(),
               d["context_lens"].data_ptr(), 2, q_len, 32, 8, 128, 16, wl.max_blocks_per_seq, wl.num_blocks,
               ctypes.c_float(wl.scale), out.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == want
    torch.cuda.synchronize()
    assert not out.any()
