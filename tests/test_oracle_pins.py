"""Pins of the CPU oracle against things other than itself.

The pages print no worked example, so the oracle is pinned by:
  * a pure-Python dense brute force over contiguous K/V (the paged result must
    equal plain softmax(q K^T scale) V -- the ForgeLLM README's "Decode-only
    block-table attention" feature promises exactly that without padded K/V);
  * torch's float64 scaled_dot_product_attention as an independent library witness;
  * invariants: permuting physical blocks, L=1, equal keys / q=0 / scale=0,
    constant V, one dominant key, GQA == MHA with repeated kv heads;
  * the split over context partitions against the unsplit result;
  * hand-derived worked examples in tests/golden/worked_examples.json;
  * a numpy scatter for the append (bit-exact).
tests/test_oracle_mutants.py checks that plausible mistakes planted in the
oracle source fail at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import dense
from tests.helpers import gather_kv, numpy_scatter, q_f64
from workloads import BF16_NAN, bf16_bits_to_f32, f32_to_bf16_bits, make_config, make_workload

HERE = os.path.dirname(os.path.abspath(__file__))


def small(S=3, Hq=4, Hkv=2, D=64, bs=16, lengths=(1, 17, 40), seed=11, pool_scale=2, **kw):
    return make_workload("small", S, Hq, Hkv, D, bs, list(lengths), seed, pool_scale=pool_scale, **kw)


def brute(wl, i, h, scale=None):
    K, V = gather_kv(wl, i)
    kh = h // wl.group
    q = q_f64(wl)[i, h]
    return np.array(dense.attention(list(q), K[:, kh].tolist(), V[:, kh].tolist(),
                                    wl.scale if scale is None else scale))


def run(orc, wl, **kw):
    args = dict(scale=wl.scale)
    args.update(kw)
    return orc.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, **args)


# --------------------------------------------------------------- brute force

def test_config1_matches_dense_bruteforce(oracle_lib):
    wl = make_config(1)
    out = run(oracle_lib, wl)
    for i in range(wl.num_seqs):
        for h in range(wl.num_q_heads):
            np.testing.assert_allclose(out[i, h], brute(wl, i, h), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Hq,Hkv,D,bs,lengths", [
    (1, 1, 64, 16, (15, 16, 17)),
    (2, 1, 64, 32, (31, 32, 33)),
    (8, 2, 128, 16, (1, 9)),
    (8, 1, 64, 16, (5, 48)),
    (4, 4, 128, 32, (3, 65)),
])
def test_edge_shapes_match_dense_bruteforce(oracle_lib, Hq, Hkv, D, bs, lengths):
    wl = small(S=len(lengths), Hq=Hq, Hkv=Hkv, D=D, bs=bs, lengths=lengths, seed=D + bs + Hq)
    out = run(oracle_lib, wl)
    for i in range(wl.num_seqs):
        for h in range(wl.num_q_heads):
            np.testing.assert_allclose(out[i, h], brute(wl, i, h), rtol=1e-12, atol=1e-13)


def test_scale_enters_scores(oracle_lib):
    wl = small(seed=5)
    for scale in (0.03, 0.5):
        out = run(oracle_lib, wl, scale=scale)
        np.testing.assert_allclose(out[2, 3], brute(wl, 2, 3, scale=scale), rtol=1e-12, atol=1e-13)


def test_torch_float64_sdpa_witness(oracle_lib):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    wl = make_config(2)
    out = run(oracle_lib, wl)
    q = torch.from_numpy(q_f64(wl))
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(wl.group, dim=0)  # [Hq, L, D]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(wl.group, dim=0)
        ref = F.scaled_dot_product_attention(q[i][:, None, :], Kt, Vt, scale=wl.scale)[:, 0, :]
        np.testing.assert_allclose(out[i], ref.numpy(), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_block_permutation_invariance_bit_identical(oracle_lib):
    wl = make_config(2)
    base = run(oracle_lib, wl)
    rng = np.random.default_rng(1)
    perm = rng.permutation(wl.num_blocks)            # block b moves to perm[b]
    kc = np.empty_like(wl.k_cache)
    vc = np.empty_like(wl.v_cache)
    kc[perm] = wl.k_cache
    vc[perm] = wl.v_cache
    tables = wl.block_tables.copy()
    nblk = (wl.context_lens + wl.block_size - 1) // wl.block_size
    for i in range(wl.num_seqs):
        tables[i, :nblk[i]] = perm[tables[i, :nblk[i]]]
    out = oracle_lib.paged_attention(wl.q, kc, vc, tables, wl.context_lens, wl.scale)
    assert np.array_equal(out, base)


def test_length_one_returns_v_exactly(oracle_lib):
    wl = small(lengths=(1, 1, 1), Hq=8, Hkv=2, seed=3)
    out = run(oracle_lib, wl)
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        for h in range(wl.num_q_heads):
            assert np.array_equal(out[i, h], V[0, h // wl.group])


def _mean_v(wl):
    ref = np.zeros((wl.num_seqs, wl.num_q_heads, wl.head_dim))
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        for h in range(wl.num_q_heads):
            ref[i, h] = V[:, h // wl.group].mean(axis=0)
    return ref


def test_zero_query_and_zero_scale_give_mean_v(oracle_lib):
    wl = small(lengths=(7, 33, 64), seed=4)
    np.testing.assert_allclose(run(oracle_lib, wl, scale=0.0), _mean_v(wl), rtol=0, atol=1e-14)
    wl.q[:] = 0
    np.testing.assert_allclose(run(oracle_lib, wl), _mean_v(wl), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_v(oracle_lib):
    wl = small(lengths=(5, 21, 40), seed=6)
    used = np.unique(wl.block_tables[wl.block_tables >= 0])
    used = used[used < wl.num_blocks]
    wl.k_cache[used] = wl.k_cache[used[0], :, :1, :]       # every key row equal (per kv head)
    np.testing.assert_allclose(run(oracle_lib, wl), _mean_v(wl), rtol=0, atol=1e-13)


def test_constant_v_gives_constant(oracle_lib):
    wl = small(lengths=(3, 30, 64), seed=7)
    c = f32_to_bf16_bits(np.array([-1.375], dtype=np.float32))[0]
    used = np.unique(wl.block_tables[(wl.block_tables >= 0) & (wl.block_tables < wl.num_blocks)])
    for i in range(wl.num_seqs):      # only valid tokens: tails stay NaN-poisoned
        L = int(wl.context_lens[i])
        for t in range(L):
            wl.v_cache[wl.block_tables[i, t // wl.block_size], :, t % wl.block_size, :] = c
    out = run(oracle_lib, wl)
    np.testing.assert_allclose(out, -1.375, rtol=0, atol=1e-15)
    assert used.size


def test_dominant_key_selects_its_value(oracle_lib):
    wl = small(S=1, Hq=2, Hkv=1, lengths=(40,), seed=8)
    tables = wl.block_tables
    j = 23                                              # the dominant token
    for t in range(40):
        wl.k_cache[tables[0, t // 16], 0, t % 16, :] = 0
    wl.k_cache[tables[0, j // 16], 0, j % 16, :] = wl.q[0, 0]
    # s_j = 20*|q|^2 (about 1300) against 0 for the others: exp(-s_j) underflows to 0, so the
    # output is V_j exactly -- and exp(s_j) overflows unless the running maximum is subtracted
    out = run(oracle_lib, wl, scale=20.0)
    K, V = gather_kv(wl, 0)
    assert np.array_equal(out[0, 0], V[j, 0])


def test_gqa_equals_mha_with_repeated_kv_heads(oracle_lib):
    wl = small(Hq=8, Hkv=2, lengths=(9, 40, 64), seed=9)
    gqa = run(oracle_lib, wl)
    g = wl.group
    kc = np.repeat(wl.k_cache, g, axis=1)               # kv head kh -> q heads kh*g .. kh*g+g-1
    vc = np.repeat(wl.v_cache, g, axis=1)
    mha = oracle_lib.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    assert np.array_equal(gqa, mha)


def test_zero_length_gives_zeros(oracle_lib):
    wl = small(lengths=(0, 17, 3), seed=10)
    out = run(oracle_lib, wl)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    np.testing.assert_allclose(out[1, 0], brute(wl, 1, 0), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ split-K

@pytest.mark.parametrize("P", [16, 32, 48, 512, 4096])
def test_split_equals_unsplit(oracle_lib, P):
    wl = small(S=4, Hq=4, Hkv=2, lengths=(1, 100, 513, 600), seed=12)
    full = run(oracle_lib, wl)
    split = oracle_lib.split_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                       wl.scale, P)
    np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-14)


def test_partition_partials_are_dense_attention_over_the_partition(oracle_lib):
    wl = small(S=2, Hq=2, Hkv=1, lengths=(70, 33), seed=13)
    P = 32
    o, m, l = oracle_lib.partition(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                   wl.scale, P)
    q = q_f64(wl)
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        L = int(wl.context_lens[i])
        for h in range(wl.num_q_heads):
            for k in range(o.shape[2]):
                t0, t1 = k * P, min((k + 1) * P, L)
                if t1 <= t0:
                    assert m[i, h, k] == -np.inf and l[i, h, k] == 0 and not o[i, h, k].any()
                    continue
                s = [wl.scale * float(np.dot(q[i, h], K[t, 0])) for t in range(t0, t1)]
                assert m[i, h, k] == pytest.approx(max(s), rel=1e-14, abs=1e-14)
                assert l[i, h, k] == pytest.approx(sum(math.exp(x - max(s)) for x in s), rel=1e-13)
                ref = dense.attention(list(q[i, h]), K[t0:t1, 0].tolist(), V[t0:t1, 0].tolist(), wl.scale)
                np.testing.assert_allclose(o[i, h, k], ref, rtol=1e-12, atol=1e-13)


def test_single_partition_merge_is_identity(oracle_lib):
    wl = small(lengths=(5, 17, 40), seed=14)
    o, m, l = oracle_lib.partition(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                   wl.scale, 64)
    assert o.shape[2] == 1
    out = oracle_lib.merge(o, m, l, wl.context_lens, 64)
    assert np.array_equal(out, o[:, :, 0, :])


# ------------------------------------------------------------ worked examples

def _load_examples():
    with open(os.path.join(HERE, "golden", "worked_examples.json")) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", _load_examples(), ids=lambda e: e["name"])
def test_worked_examples(oracle_lib, ex):
    """Hand-derived single-sequence cases; every input is exactly representable in bf16."""
    q = np.array(ex["q"], dtype=np.float32)              # [Hq, D]
    K = np.array(ex["K"], dtype=np.float32)              # [L, Hkv, D]
    V = np.array(ex["V"], dtype=np.float32)
    Hq, D = q.shape
    L, Hkv, _ = K.shape
    bs = ex["block_size"]
    nb = (L + bs - 1) // bs
    order = ex["table"]                                  # physical block of each logical block
    NB = max(order) + 1
    kc = np.full((NB, Hkv, bs, D), BF16_NAN, dtype=np.uint16)
    vc = kc.copy()
    for t in range(L):
        kc[order[t // bs], :, t % bs, :] = f32_to_bf16_bits(K[t])
        vc[order[t // bs], :, t % bs, :] = f32_to_bf16_bits(V[t])
    qb = f32_to_bf16_bits(q)[None]
    assert np.array_equal(bf16_bits_to_f32(qb[0]), q)    # inputs are exact
    out = oracle_lib.paged_attention(qb, kc, vc, np.array([order[:nb]], dtype=np.int32),
                                     np.array([L], dtype=np.int32), ex["scale"])
    np.testing.assert_allclose(out[0], np.array(ex["expected"]), rtol=1e-14, atol=1e-15)


# -------------------------------------------------------------------- append

def test_append_matches_numpy_scatter_bit_exact(oracle_lib):
    wl = make_config(3)
    kc, vc, bad = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                               wl.block_size)
    rk, rv = numpy_scatter(wl)
    assert bad == 0
    assert np.array_equal(kc, rk) and np.array_equal(vc, rv)
    # the -1 rows changed nothing: the only changed rows are the valid slots
    changed = np.argwhere((kc != wl.k_cache).any(axis=(1, 3)))
    assert len({(int(b), int(h)) for b, h in changed}) <= int((wl.slot_mapping >= 0).sum()) * wl.num_kv_heads


def test_append_skips_minus_one_and_counts_out_of_range(oracle_lib):
    wl = small(S=4, lengths=(4, 17, 30, 2), seed=15, append=True)
    sentinel_k = np.full_like(wl.k_cache, 0x1234)
    sentinel_v = np.full_like(wl.v_cache, 0x4321)
    slots = wl.slot_mapping.copy()
    slots[1] = -1
    slots[2] = -7                                        # out of range: skipped, counted
    slots[3] = wl.num_blocks * wl.block_size             # out of range
    kc, vc, bad = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, slots, sentinel_k, sentinel_v,
                                               wl.block_size)
    assert bad == 2
    s = int(slots[0])
    exp_k, exp_v = sentinel_k.copy(), sentinel_v.copy()
    exp_k[s // wl.block_size, :, s % wl.block_size, :] = wl.new_k[0]
    exp_v[s // wl.block_size, :, s % wl.block_size, :] = wl.new_v[0]
    assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


def test_append_then_attend_sees_new_token(oracle_lib):
    wl = make_config(3)
    kc, vc, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                             wl.block_size)
    out = oracle_lib.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    assert np.all(np.isfinite(out))                      # no poisoned (unfilled) slot was read
    before = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                        wl.scale)
    appended = wl.slot_mapping >= 0
    assert np.all(np.isnan(before[appended]).any(axis=(1, 2)))
    assert np.all(np.isfinite(before[~appended]))


# ---------------------------------------------------------------- block copy

def _copy_case(seed=16):
    wl = small(S=3, Hq=8, Hkv=2, D=64, bs=16, lengths=(20, 40, 33), seed=seed, pool_scale=3)
    rng = np.random.default_rng(seed)
    used = np.unique(wl.block_tables[(wl.block_tables >= 0) & (wl.block_tables < wl.num_blocks)])
    free = np.setdiff1d(np.arange(wl.num_blocks), used)
    src = rng.choice(used, size=4, replace=False)
    dst = rng.choice(free, size=4, replace=False)
    return wl, np.stack([src, dst], axis=1)


def test_copy_blocks_matches_numpy_bit_exact(oracle_lib):
    wl, pairs = _copy_case()
    kc, vc, bad = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, pairs)
    ek, ev = wl.k_cache.copy(), wl.v_cache.copy()
    ek[pairs[:, 1]] = wl.k_cache[pairs[:, 0]]
    ev[pairs[:, 1]] = wl.v_cache[pairs[:, 0]]
    assert bad == 0 and np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_copy_blocks_identity_and_out_of_range(oracle_lib):
    wl, pairs = _copy_case(17)
    same = np.stack([pairs[:, 0], pairs[:, 0]], axis=1)
    kc, vc, bad = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, same)
    assert bad == 0 and np.array_equal(kc, wl.k_cache) and np.array_equal(vc, wl.v_cache)
    broken = np.array([[-1, pairs[0, 1]], [pairs[1, 0], wl.num_blocks], [pairs[2, 0], pairs[2, 1]]])
    kc, vc, bad = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, broken)
    ek = wl.k_cache.copy()
    ek[pairs[2, 1]] = wl.k_cache[pairs[2, 0]]
    assert bad == 2 and np.array_equal(kc, ek)


def test_forked_sequence_attends_like_its_parent(oracle_lib):
    """A fork copies the parent's last block into a fresh one and rewrites its table entry."""
    wl, pairs = _copy_case(18)
    i = 1
    nb = int((wl.context_lens[i] + wl.block_size - 1) // wl.block_size)
    last = wl.block_tables[i, nb - 1]
    fresh = np.setdiff1d(np.arange(wl.num_blocks), wl.block_tables[wl.block_tables >= 0])[0]
    kc, vc, _ = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, [[last, fresh]])
    tables = wl.block_tables.copy()
    tables[i, nb - 1] = fresh
    a = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    b = oracle_lib.paged_attention(wl.q, kc, vc, tables, wl.context_lens, wl.scale)
    assert np.array_equal(a, b)


# --------------------------------------------------------- multi-token query

def _multi(wl, Q):
    from workloads import multi_query
    return multi_query(wl, Q)


def test_multi_query_single_token_is_decode(oracle_lib):
    wl = small(S=3, Hq=8, Hkv=2, lengths=(5, 40, 64), seed=19)
    q = wl.q[:, None]                                        # [S, 1, Hq, D]
    m = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    assert np.array_equal(m[:, 0], run(oracle_lib, wl))


def test_multi_query_rows_are_decodes_of_their_prefix(oracle_lib):
    """Row j of sequence i equals a decode of query q[i, j] over the first L_i - Q + j + 1 tokens."""
    wl = small(S=3, Hq=4, Hkv=2, lengths=(9, 33, 60), seed=20)
    Q = 5
    q = _multi(wl, Q)
    m = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    for j in range(Q):
        lens = (wl.context_lens - Q + j + 1).astype(np.int32)
        ref = oracle_lib.paged_attention(q[:, j], wl.k_cache, wl.v_cache, wl.block_tables, lens, wl.scale)
        assert np.array_equal(m[:, j], ref)


def test_multi_query_long_draft_rows_are_decodes_of_their_prefix(oracle_lib):
    """The same property with 16 new tokens at g = 4 (64 query rows per kv head, the widest the
    GPU kernels take) and a sequence shorter than the draft (its first rows are zero)."""
    wl = small(S=3, Hq=8, Hkv=2, lengths=(12, 70, 129), seed=22)
    Q = 16
    q = _multi(wl, Q)
    m = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    for j in range(Q):
        lens = np.maximum(wl.context_lens - Q + j + 1, 0).astype(np.int32)
        ref = oracle_lib.paged_attention(q[:, j], wl.k_cache, wl.v_cache, wl.block_tables, lens, wl.scale)
        assert np.array_equal(m[:, j], ref)
    assert not m[0, :4].any()


def test_multi_query_dense_bruteforce_causal(oracle_lib):
    wl = small(S=2, Hq=4, Hkv=1, D=64, lengths=(7, 20), seed=21)
    Q = 4
    q = _multi(wl, Q)
    m = oracle_lib.paged_attention_multi(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    for i in range(wl.num_seqs):
        K, V = gather_kv(wl, i)
        L = int(wl.context_lens[i])
        for j in range(Q):
            pos = L - Q + j
            for h in range(wl.num_q_heads):
                ref = dense.attention(list(qf[i, j, h]), K[:pos + 1, 0].tolist(), V[:pos + 1, 0].tolist(), wl.scale)
                np.testing.assert_allclose(m[i, j, h], ref, rtol=1e-12, atol=1e-13)


def test_multi_query_rows_before_the_sequence_start_are_zero(oracle_lib):
    wl = small(S=2, Hq=2, Hkv=1, lengths=(2, 30), seed=22)
    Q = 4                                                     # sequence 0 has only 2 tokens
    m = oracle_lib.paged_attention_multi(_multi(wl, Q), wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                         wl.scale)
    assert not m[0, :2].any() and np.all(np.isfinite(m[0, 2:])) and m[0, 2:].any()
