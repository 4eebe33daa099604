"""Seeded random shapes through every attention entry point, against the fp64 oracle.

Each case draws a head layout (g in {1, 2, 4, 8}), head_dim, block size (16, 32 or 48),
sequence count and lengths (empty and one-token sequences included, lengths on and off
16-token tiles) from its own seed, and checks on that one workload: the single pass, the
bf16-output single pass, the fixed-partition split at a random partition size, the auto
decode (whichever of its plans the sizes select), and the multi-token query at a few
q_len values (16-row, wide, tcgen05 and prompt-chunk kernels, as the rows fall).  Small
sizes keep the oracle to a fraction of a second per case.
"""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import bf16_bits_to_f32, make_workload, multi_query

pytestmark = pytest.mark.gpu


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    g = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 48]))
    S = int(rng.integers(1, 13))
    kind = rng.random(S)
    lengths = np.where(kind < 0.1, 0, np.where(kind < 0.2, 1, rng.integers(2, 2500, S)))
    return g * Hkv, Hkv, D, bs, [int(x) for x in lengths]


@pytest.mark.parametrize("seed", range(64))
def test_random_shapes_all_entry_points(pf, oracle_lib, seed):
    Hq, Hkv, D, bs, lengths = draw_case(seed)
    wl = make_workload("rand", len(lengths), Hq, Hkv, D, bs, lengths, seed=2000 + seed, pool_scale=2)
    d = to_device(wl)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    mx = max(int(wl.max_context_len), 16)
    rng = np.random.default_rng(3000 + seed)
    P = int(rng.choice([16, 64, 256, 512, 1024]))

    outs = {
        "decode": pf.paged_attention_decode(*attn_args(d)),
        "split": pf.paged_attention_split(*attn_args(d), partition_size=P, max_context_len=mx),
        "auto": pf.paged_attention_decode_auto(*attn_args(d), max_context_len=mx),
    }
    b16 = pf.paged_attention_decode_bf16(*attn_args(d))
    assert pf.get_device_error() == pf.PF_OK, (Hq, Hkv, D, bs, lengths)
    for name, out in outs.items():
        check_close(out.cpu().numpy(), ref)
    got16 = bf16_bits_to_f32(b16.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    assert np.all(np.abs(got16 - ref) <= 2e-3 + 1e-2 * np.abs(ref)), "bf16 output"
    for i, L in enumerate(lengths):
        if L == 0:
            assert not outs["decode"][i].any() and not outs["auto"][i].any()

    # multi-token queries: q_len chosen so that the rows per kv head land in different kernels
    g = Hq // Hkv
    for q_len in sorted({1, max(1, 16 // g), max(1, 48 // g), max(1, 160 // g)}):
        q = multi_query(wl, q_len)
        qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).view(torch.bfloat16).cuda()
        got = pf.paged_attention_multi_query(qt, *attn_args(d)[1:]).cpu().numpy()
        assert pf.get_device_error() == pf.PF_OK, (Hq, Hkv, D, bs, lengths, q_len)
        refm = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                                wl.scale)
        check_close(got, refm)
