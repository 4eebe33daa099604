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
