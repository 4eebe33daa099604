"""The split-K entry point that allocates nothing (pf_paged_attention_split_noalloc).

It is meant for callers that cannot allocate device memory when they decode --
a plugin whose host runtime owns all device memory, a loop that must not call
cudaMalloc because it can stall the whole device, a process whose memory another
allocator has already taken.  Its partials live in a fixed scratch array inside
the library, shared by every call on a device.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def _noalloc_call(pf, d, wl, P, max_ctx, out):
    f = pf.lib().pf_paged_attention_split_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    q, kc, vc, bt, cl = attn_args(d)
    return f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(), wl.num_seqs,
             wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.max_blocks_per_seq, wl.num_blocks,
             wl.scale, P, max_ctx, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_split_on_two_calls_in_a_row(pf):
    cases = [
        (make_workload("na1", 6, 32, 8, 128, 16, [3000, 17, 512, 1, 2048, 900], seed=61), 512),
        (make_workload("na2", 3, 16, 2, 64, 32, [700, 65, 1500], seed=62, pool_scale=2), 128),
    ]
    for wl, P in cases:                  # the second call finds the first call's partials in the scratch
        d = to_device(wl)
        max_ctx = wl.max_context_len
        want = pf.paged_attention_split(*attn_args(d), partition_size=P, max_context_len=max_ctx)
        got = torch.full_like(want, float("nan"))
        assert _noalloc_call(pf, d, wl, P, max_ctx, got) == pf.PF_OK
        assert pf.get_device_error() == pf.PF_OK
        check_close(got.cpu().numpy(), want.cpu().numpy())


def test_noalloc_rejects_sizes_beyond_its_scratch(pf):
    wl = make_workload("big", 2, 32, 8, 128, 16, [64, 64], seed=63)
    d = to_device(wl)
    out = torch.zeros((2, 32, 128), dtype=torch.float32, device="cuda")
    huge = 1 << 20        # 2 x 32 heads x 2048 partitions of 16 tokens: far beyond 16 MiB of partials
    assert pf.partition_workspace_layout(2, 32, 128, huge, 16)[0] > pf.SPLIT_NOALLOC_SCRATCH_BYTES
    assert _noalloc_call(pf, d, wl, 16, huge, out) == pf.PF_ERR_UNSUPPORTED
    assert not out.any()
