"""Persistent single-pass decode (resident CTAs taking items longest first from a work
counter in the caller's workspace) on the GPU.

Each item runs the arithmetic of pf_paged_attention_decode, so the outputs are compared
with that call's bit for bit, and with the fp64 oracle within the attention tolerance.
The workspace cases cover the counter protocol: any initial contents, reuse by later
calls, reuse after another call wrote into it, and replays of a captured launch.
"""
import numpy as np
import pytest
import torch

import dataclasses

from tests.helpers import attn_args, check_close, numpy_scatter, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def persistent(pf, d, ws=None, **kw):
    out = pf.paged_attention_decode_persistent(*attn_args(d), workspace=ws, **kw)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


def single(pf, d, **kw):
    out = pf.paged_attention_decode(*attn_args(d), **kw)
    assert pf.get_device_error() == pf.PF_OK
    return out.cpu().numpy()


def oracle_out(orc, wl):
    return orc.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)


def appended(pf, wl):
    """The workload after its append (device tensors, and the numpy workload for the oracle);
    before it, the slots about to be filled hold NaN."""
    d = to_device(wl)
    if wl.slot_mapping is not None:
        pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
        kc, vc = numpy_scatter(wl)
        wl = dataclasses.replace(wl, k_cache=kc, v_cache=vc)
    return d, wl


def workspace(fill=None):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    if fill is not None:
        ws.copy_(torch.from_numpy(np.frombuffer(fill, dtype=np.uint8).copy()))
    return ws


@pytest.mark.parametrize("index", [1, 2, 3])
def test_named_workloads(pf, oracle_lib, config_workload, index):
    d, wl = appended(pf, config_workload(index))
    got = persistent(pf, d)
    check_close(got, oracle_out(oracle_lib, wl))
    assert np.array_equal(got, single(pf, d))


def test_llama3_8b_full_size(pf, oracle_lib, config_workload):
    """The bench's workload: every row equal to the one-CTA-per-item decode, sampled rows
    and every head of the longest sequence against the oracle."""
    wl = config_workload(4)
    d = to_device(wl)
    got = persistent(pf, d)
    assert np.array_equal(got, single(pf, d))
    rng = np.random.default_rng(321)
    pairs = [(int(rng.integers(wl.num_seqs)), int(rng.integers(wl.num_q_heads))) for _ in range(32)]
    longest = int(np.argmax(wl.context_lens))
    pairs += [(longest, h) for h in range(0, wl.num_q_heads, 2)]
    ref = oracle_lib.paged_attention_pairs(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                                           wl.scale, pairs)
    check_close(np.stack([got[i, h] for i, h in pairs]), ref)
    del d
    torch.cuda.empty_cache()


EDGE_LENGTHS = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 0]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_edge_lengths_all_variants(pf, oracle_lib, D, bs, g):
    Hkv = 2
    wl = make_workload("pedge", len(EDGE_LENGTHS), Hkv * g, Hkv, D, bs, EDGE_LENGTHS,
                       seed=D * 100 + bs * 10 + g + 7, pool_scale=2)
    d = to_device(wl)
    got = persistent(pf, d)
    check_close(got, oracle_out(oracle_lib, wl))
    assert np.array_equal(got, single(pf, d))


@pytest.mark.parametrize("D,g", [(128, 1), (64, 4)])
def test_many_short_items_take_the_counter_path(pf, oracle_lib, D, g):
    """512 sequences (the limit) x 8 kv heads = 4,096 items, many more than two per resident
    CTA, mostly short and some empty: most items come from the work counter."""
    rng = np.random.default_rng(40 + D)
    lens = np.minimum(np.round(np.exp(rng.uniform(0, np.log(600), 512))), 600).astype(np.int64)
    lens[rng.choice(512, 40, replace=False)] = 0
    wl = make_workload("pmany", 512, 8 * g, 8, D, 16, lens.tolist(), seed=50 + D)
    d = to_device(wl)
    got = persistent(pf, d)
    check_close(got, oracle_out(oracle_lib, wl))
    assert np.array_equal(got, single(pf, d))


def test_workspace_contents_do_not_matter(pf, config_workload):
    """Garbage, zeros, and a counter that looks like a finished call: all give the same output,
    and every call leaves the two counters at zero."""
    d, _ = appended(pf, config_workload(3))
    ref = single(pf, d)
    rng = np.random.default_rng(5)
    stale = np.zeros(32, dtype=np.uint64)
    other = np.uint64(0xDEADBEEF) << np.uint64(32)                  # an epoch no call here reaches
    stale[0] = other | np.uint64(10 ** 6)                            # counted far past the end
    stale[1] = other | np.uint64(3)
    for fill in (rng.integers(0, 256, 256, dtype=np.uint8).tobytes(), bytes(256), stale.tobytes()):
        ws = workspace(fill)
        for _ in range(2):  # the second call finds the counters the first one cleared
            assert np.array_equal(persistent(pf, d, ws), ref)
            assert not ws[:16].cpu().numpy().any()


def test_workspace_shared_with_the_split(pf, config_workload):
    """A workspace whose first bytes the partition pass filled with partials."""
    wl = config_workload(2)
    d = to_device(wl)
    ref = single(pf, d)
    P, mx = 64, wl.max_context_len
    ws = pf.alloc_workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, mx, P, "cuda")
    pf.paged_attention_decode_partition(*attn_args(d), P, mx, ws)
    assert pf.get_device_error() == pf.PF_OK
    assert ws[:16].cpu().numpy().any()
    assert np.array_equal(persistent(pf, d, ws[:256]), ref)


def test_graph_replays(pf, config_workload):
    """One captured launch replayed with new queries: the counters the previous replay
    cleared serve the next one (the launch's epoch is fixed at capture)."""
    d, wl = appended(pf, config_workload(3))
    ws = workspace()
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    pf.paged_attention_decode_persistent(*attn_args(d), workspace=ws, out=out)  # first call outside capture
    torch.cuda.synchronize()
    q_static = d["q"]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pf.paged_attention_decode_persistent(*attn_args(d), workspace=ws, out=out)
    torch.cuda.current_stream().wait_stream(s)
    rng = np.random.default_rng(9)
    for r in range(3):
        q_new = torch.from_numpy(rng.standard_normal(tuple(q_static.shape)).astype(np.float32)).to(
            "cuda", torch.bfloat16)
        q_static.copy_(q_new)
        g.replay()
        torch.cuda.synchronize()
        assert pf.get_device_error() == pf.PF_OK
        assert np.array_equal(out.cpu().numpy(), single(pf, d)), f"replay {r}"


def test_bad_length_and_block_give_nan_rows(pf):
    wl = make_workload("pbad", 4, 8, 2, 128, 16, [40, 70, 33, 20], seed=61, pool_scale=2)
    d = to_device(wl)
    d["context_lens"][1] = wl.block_tables.shape[1] * wl.block_size + 1   # beyond the table
    d["block_tables"][2, 1] = wl.num_blocks + 5                            # block id out of range
    out = pf.paged_attention_decode_persistent(*attn_args(d)).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(out[1]).all() and np.isnan(out[2]).all()
    assert np.isfinite(out[0]).all() and np.isfinite(out[3]).all()


def test_deterministic_and_stream_ordered(pf, config_workload):
    d, _ = appended(pf, config_workload(3))
    ws = workspace()
    a = persistent(pf, d, ws)
    outs = [pf.paged_attention_decode_persistent(*attn_args(d), workspace=ws) for _ in range(5)]
    assert pf.get_device_error() == pf.PF_OK
    for o in outs:
        assert np.array_equal(o.cpu().numpy(), a)
