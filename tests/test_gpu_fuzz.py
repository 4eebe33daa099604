"""Seeded random shapes through every attention entry point against the oracle: group
sizes 1-8, head dims 64/128, block sizes 16-64, lengths from 0 to a few hundred with tile
and block boundaries over-represented, partition sizes 16-512 and multi-token queries
up to the 64-row limit."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload, multi_query

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    g = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 48, 64]))
    S = int(rng.integers(1, 24))
    lens = []
    for _ in range(S):
        kind = rng.integers(4)
        if kind == 0:
            lens.append(int(rng.integers(0, 3)))
        elif kind == 1:
            lens.append(int(16 * rng.integers(1, 20) + rng.integers(-1, 2)))
        else:
            lens.append(int(rng.integers(1, 400)))
    return rng, g, Hkv, D, bs, S, [max(0, x) for x in lens]


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(pf, oracle_lib, seed):
    rng, g, Hkv, D, bs, S, lens = _case(seed)
    wl = make_workload("fuzz", S, g * Hkv, Hkv, D, bs, lens, seed=2000 + seed, pool_scale=2, append=True,
                       num_skip_slots=int(rng.integers(0, 2)) if S > 1 else 0)
    d = to_device(wl)
    # fused append + decode, then the split and the plain decode over the appended cache
    got = pf.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"],
                                           d["v_cache"], d["block_tables"], d["context_lens"]).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    kc, vc, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                             wl.block_size)
    ref = oracle_lib.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got, ref)
    single = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    assert np.array_equal(single, got)
    P = int(rng.choice([16, 32, 64, 128, 512]))
    mx = max(1, int(max(lens)))
    split = pf.paged_attention_split(*attn_args(d), partition_size=P, max_context_len=mx).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    check_close(split, ref)
    # several new tokens per sequence over the appended cache
    q_len = int(rng.integers(1, 64 // g + 1))
    q = multi_query(wl, q_len)
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
    mq_ref = oracle_lib.paged_attention_multi(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    for kernel in ("auto", "tcgen05") if wl.head_dim == 128 else ("auto",):
        mq = pf.paged_attention_multi_query(qt, d["k_cache"], d["v_cache"], d["block_tables"],
                                            d["context_lens"], kernel=kernel).cpu().numpy()
        assert pf.get_device_error() == pf.PF_OK
        check_close(mq, mq_ref)
