"""The split-K entry point that allocates nothing (pf_paged_attention_split_noalloc).

It is meant for callers that cannot allocate device memory when they decode --
a plugin whose host runtime owns all device memory, a loop that must not call
cudaMalloc because it can stall the whole device, a process whose memory another
allocator has already taken.  Its partials live in a fixed scratch array inside
the library, shared by every call on a device.

The entry point runs the same partition pass and merge as the workspace split
with the same arguments, so its output must be bit-identical to that split's;
any difference would mean a wrong scratch address or a stale partial.  It is
also checked against the fp64 oracle within the attention tolerance.

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


def _noalloc_fn(pf):
    f = pf.lib().pf_paged_attention_split_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _noalloc_call(pf, d, wl, P, max_ctx, out, num_q_heads=None, num_kv_heads=None):
    q, kc, vc, bt, cl = attn_args(d)
    hq = wl.num_q_heads if num_q_heads is None else num_q_heads
    hkv = wl.num_kv_heads if num_kv_heads is None else num_kv_heads
    return _noalloc_fn(pf)(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(), wl.num_seqs,
                           hq, hkv, wl.head_dim, wl.block_size, wl.max_blocks_per_seq, wl.num_blocks, wl.scale, P,
                           max_ctx, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _check_case(pf, oracle_lib, wl, P, max_ctx):
    """One no-allocation call: bit-identical to the workspace split, within tolerance of the oracle."""
    d = to_device(wl)
    want = pf.paged_attention_split(*attn_args(d), partition_size=P, max_context_len=max_ctx)
    got = torch.full_like(want, float("nan"))
    assert _noalloc_call(pf, d, wl, P, max_ctx, got) == pf.PF_OK
    assert pf.get_device_error() == pf.PF_OK
    assert torch.equal(got, want)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_close(got.cpu().numpy(), ref)
    return got


# 11 sequences x 7 query heads x 419 partitions of 128 dims: 512 * 32,263 bytes of
# o_k plus two 256-byte-rounded m_k / l_k arrays of 129,280 bytes is exactly 16 MiB.
EDGE_SEQS, EDGE_HEADS, EDGE_P, EDGE_NP = 11, 7, 16, 419


def _edge_workload():
    rng = np.random.Generator(np.random.PCG64(64))
    lens = rng.integers(1, 700, size=EDGE_SEQS).astype(np.int32)
    lens[-1] = EDGE_NP * EDGE_P            # the last sequence writes the scratch's last partials
    lens[3] = EDGE_NP * EDGE_P - 5
    return make_workload("na_edge", EDGE_SEQS, EDGE_HEADS, EDGE_HEADS, 128, 16, lens, seed=64)


def test_noalloc_matches_workspace_split_and_oracle_on_two_calls_in_a_row(pf, oracle_lib):
    cases = [
        (make_workload("na1", 6, 32, 8, 128, 16, [3000, 17, 512, 1, 2048, 900], seed=61), 512),
        (make_workload("na2", 3, 16, 2, 64, 32, [700, 65, 1500], seed=62, pool_scale=2), 128),
    ]
    for wl, P in cases:                  # the second call finds the first call's partials in the scratch
        _check_case(pf, oracle_lib, wl, P, wl.max_context_len)


def test_noalloc_layout_exactly_at_the_scratch_size(pf, oracle_lib):
    max_ctx = EDGE_NP * EDGE_P
    need = pf.partition_workspace_layout(EDGE_SEQS, EDGE_HEADS, 128, max_ctx, EDGE_P)[0]
    assert need == pf.SPLIT_NOALLOC_SCRATCH_BYTES
    _check_case(pf, oracle_lib, _edge_workload(), EDGE_P, max_ctx)


def test_noalloc_layout_one_partition_over_the_scratch_size(pf):
    wl = _edge_workload()
    max_ctx = EDGE_NP * EDGE_P + 1          # one more partition per row: 420
    assert pf.partition_workspace_layout(EDGE_SEQS, EDGE_HEADS, 128, max_ctx, EDGE_P)[0] > \
        pf.SPLIT_NOALLOC_SCRATCH_BYTES
    d = to_device(wl)
    out = torch.zeros((EDGE_SEQS, EDGE_HEADS, 128), dtype=torch.float32, device="cuda")
    assert _noalloc_call(pf, d, wl, EDGE_P, max_ctx, out) == pf.PF_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not out.any()


def test_noalloc_empty_sequence_after_a_large_call_reads_no_stale_partial(pf, oracle_lib):
    # fill the whole scratch with finite partials first ...
    _check_case(pf, oracle_lib, _edge_workload(), EDGE_P, EDGE_NP * EDGE_P)
    # ... then a small layout whose m_k / l_k arrays start inside the old o_k region
    wl = make_workload("na_small", 4, 8, 2, 128, 16, [0, 40, 300, 0], seed=65)
    got = _check_case(pf, oracle_lib, wl, 32, wl.max_context_len)
    assert not got[0].any() and not got[3].any()


def test_noalloc_rejects_sizes_beyond_its_scratch(pf):
    wl = make_workload("big", 2, 32, 8, 128, 16, [64, 64], seed=63)
    d = to_device(wl)
    out = torch.zeros((2, 32, 128), dtype=torch.float32, device="cuda")
    huge = 1 << 20        # 65,536 partitions of 16 tokens x 2 sequences x 32 heads: 2 GiB of o_k alone
    assert pf.partition_workspace_layout(2, 32, 128, huge, 16)[0] > pf.SPLIT_NOALLOC_SCRATCH_BYTES
    assert _noalloc_call(pf, d, wl, 16, huge, out) == pf.PF_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not out.any()


def test_noalloc_reports_a_bad_argument_before_the_size(pf):
    wl = make_workload("bad", 2, 32, 8, 128, 16, [64, 64], seed=63)
    d = to_device(wl)
    out = torch.zeros((2, 32, 128), dtype=torch.float32, device="cuda")
    huge = 1 << 20
    # query heads that are not a multiple of the kv heads, with a size far beyond the scratch
    assert _noalloc_call(pf, d, wl, 16, huge, out, num_q_heads=30) == pf.PF_ERR_INVALID_ARG
    # a partition size that is not a multiple of 16
    assert _noalloc_call(pf, d, wl, 24, wl.max_context_len, out) == pf.PF_ERR_UNSUPPORTED
    # a misaligned output, within the scratch size: nothing is launched
    flat = torch.zeros(2 * 32 * 128 + 1, dtype=torch.float32, device="cuda")
    q, kc, vc, bt, cl = attn_args(d)
    st = _noalloc_fn(pf)(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(), 2, 32, 8, 128,
                         16, wl.max_blocks_per_seq, wl.num_blocks, wl.scale, 16, wl.max_context_len,
                         flat.data_ptr() + 4, torch.cuda.current_stream().cuda_stream)
    assert st == pf.PF_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not flat.any()
