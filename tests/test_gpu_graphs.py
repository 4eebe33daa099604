"""The step captured in a CUDA graph and replayed: append + decode, the split (whose merge
is launched with programmatic dependent launch) and the multi-token query.  Each call is
made once eagerly first (the library's one-time per-device set-up happens there); the
replays, with new inputs copied into the captured buffers, must match eager calls."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, to_device
from workloads import make_workload, multi_query

pytestmark = pytest.mark.gpu


def test_decode_step_in_a_graph(pf):
    wl = make_workload("graph", 6, 16, 4, 128, 16, [5, 90, 300, 17, 64, 200], seed=91, pool_scale=2,
                       append=True, num_skip_slots=1)
    d = to_device(wl)
    P, mx = 64, wl.max_context_len
    ws = pf.alloc_workspace(wl.num_seqs, wl.num_q_heads, wl.head_dim, mx, P, "cuda")
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    split = torch.empty_like(out)

    def step():
        pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
        pf.paged_attention_decode(*attn_args(d), out=out)
        pf.paged_attention_decode_partition(*attn_args(d), P, mx, ws)
        pf.paged_attention_merge(ws, d["context_lens"], wl.num_q_heads, wl.head_dim, P, mx, out=split)

    step()  # eager first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    rng = np.random.default_rng(3)
    for r in range(3):
        for name in ("q", "new_k", "new_v"):
            t = d[name]
            t.copy_(torch.from_numpy(rng.standard_normal(tuple(t.shape)).astype(np.float32)).to("cuda", t.dtype))
        g.replay()
        torch.cuda.synchronize()
        assert pf.get_device_error() == pf.PF_OK
        got_out, got_split = out.clone(), split.clone()
        step()  # eager on the same (already appended) state
        torch.cuda.synchronize()
        assert torch.equal(got_out, out) and torch.equal(got_split, split), f"replay {r}"
        assert torch.isfinite(got_out).all()


def test_multi_query_in_a_graph(pf):
    wl = make_workload("graphmq", 4, 32, 8, 128, 16, [40, 100, 260, 33], seed=92, pool_scale=2)
    d = to_device(wl)
    # the 16-row kernel, the wide one and the tcgen05 form
    for q_len, kernel in ((4, "auto"), (8, "auto"), (8, "tcgen05")):
        qt = torch.from_numpy(np.ascontiguousarray(multi_query(wl, q_len)).view(np.int16)).view(
            torch.bfloat16).cuda()
        out = torch.empty((wl.num_seqs, q_len, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
        args = (qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
        pf.paged_attention_multi_query(*args, out=out, kernel=kernel)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                pf.paged_attention_multi_query(*args, out=out, kernel=kernel)
        torch.cuda.current_stream().wait_stream(s)
        qt.copy_(torch.randn(tuple(qt.shape), device="cuda").to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert pf.get_device_error() == pf.PF_OK
        got = out.clone()
        ref = pf.paged_attention_multi_query(*args, kernel=kernel)
        assert torch.equal(got, ref)


def _capture(fn):
    """fn() once eagerly, then captured on a side stream; returns the graph."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def test_auto_decode_prompt_chunk_bf16_and_fused_step_in_graphs(pf):
    """The launches the other graph tests leave out: the auto decode's cluster split (a cluster
    launch) and its workspace split, the prompt-chunk kernel (160 rows per kv head), the
    fused append + decode, the bf16-output decode and the block copy.  Each replay, after new
    inputs are copied into the captured buffers, is bit-identical to an eager call."""
    rng = np.random.default_rng(5)

    def refill(*ts):
        for t in ts:
            t.copy_(torch.from_numpy(rng.standard_normal(tuple(t.shape)).astype(np.float32)).to("cuda", t.dtype))

    # few items, short contexts: the cluster split; few items, one long context: the workspace split
    for lengths, want_ws in (([30, 200, 77, 512], False), ([9000, 40, 300, 5], True)):
        wl = make_workload("graphauto", 4, 16, 4, 128, 16, lengths, seed=93 + want_ws, pool_scale=2)
        d = to_device(wl)
        mx = wl.max_context_len
        P, need = pf.decode_auto_plan(4, 16, 4, 128, mx)
        assert P > 0 and (need > 0) == want_ws
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        out = torch.empty((4, 16, 128), dtype=torch.float32, device="cuda")
        g = _capture(lambda: pf.paged_attention_decode_auto(*attn_args(d), mx, workspace=ws, out=out))
        for r in range(2):
            refill(d["q"])
            g.replay()
            torch.cuda.synchronize()
            got = out.clone()
            assert torch.equal(got, pf.paged_attention_decode_auto(*attn_args(d), mx, workspace=ws)), (lengths, r)
            assert torch.isfinite(got).all()

    # the prompt-chunk kernel
    wl = make_workload("graphchunk", 3, 32, 8, 128, 16, [60, 300, 1000], seed=95, pool_scale=2)
    d = to_device(wl)
    qt = torch.from_numpy(np.ascontiguousarray(multi_query(wl, 40)).view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty((3, 40, 32, 128), dtype=torch.float32, device="cuda")
    args = (qt, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    g = _capture(lambda: pf.paged_attention_multi_query(*args, out=out))
    refill(qt)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.clone(), pf.paged_attention_multi_query(*args))

    # the fused append + decode, the bf16-output decode and a block copy in one graph
    wl = make_workload("graphfused", 5, 16, 4, 128, 16, [5, 90, 300, 17, 64], seed=96, pool_scale=2,
                       append=True, num_skip_slots=1)
    d = to_device(wl)
    out = torch.empty((5, 16, 128), dtype=torch.float32, device="cuda")
    out16 = torch.empty((5, 16, 128), dtype=torch.bfloat16, device="cuda")
    used = set(int(b) for row, L in zip(wl.block_tables, wl.context_lens) for b in row[:(int(L) + 15) // 16])
    free = [b for b in range(wl.num_blocks) if b not in used][:4]
    src = sorted(used)[:4]
    mapping = torch.tensor(list(zip(src, free)), dtype=torch.int64, device="cuda")

    def step():
        pf.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"],
                                         d["v_cache"], d["block_tables"], d["context_lens"], out=out)
        pf.paged_attention_decode_bf16(*attn_args(d), out=out16)
        pf.copy_blocks(d["k_cache"], d["v_cache"], mapping)

    g = _capture(step)
    refill(d["q"], d["new_k"], d["new_v"])
    g.replay()
    torch.cuda.synchronize()
    assert pf.get_device_error() == pf.PF_OK
    got, got16 = out.clone(), out16.clone()
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    step()  # eager on the same (already appended, already copied) state
    torch.cuda.synchronize()
    assert torch.equal(got, out) and torch.equal(got16, out16)
    bits = lambda t: t.view(torch.int16)  # the caches hold NaN poison in unused slots: compare bits
    assert torch.equal(bits(kc), bits(d["k_cache"])) and torch.equal(bits(vc), bits(d["v_cache"]))
    for s_, t_ in zip(src, free):
        assert torch.equal(bits(d["k_cache"][t_]), bits(d["k_cache"][s_]))
        assert torch.equal(bits(d["v_cache"][t_]), bits(d["v_cache"][s_]))
