"""Error paths on the GPU.  None of them faults, traps or hangs the device: bad inputs are
caught by the kernels' own range checks (the offending rows become NaN and the error word
is set), and the timeout path is driven by a wait that nothing completes."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def test_bad_block_id_flags_bounds_and_nans_only_that_item(pf, oracle_lib):
    wl = make_workload("badblk", 3, 8, 2, 128, 16, [40, 50, 60], seed=51, pool_scale=2)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    for bad in (-3, wl.num_blocks, 2 ** 31 - 1):
        d = to_device(wl)
        d["block_tables"][1, 2] = bad                  # seq 1, its last block
        out = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
        assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
        assert np.isnan(out[1]).all()                  # both kv heads of seq 1 read that block
        check_close(out[[0, 2]], ref[[0, 2]])


def test_length_beyond_table_flags_bounds(pf, oracle_lib):
    wl = make_workload("badlen", 2, 4, 2, 64, 16, [10, 20], seed=52)
    d = to_device(wl)
    d["context_lens"][0] = wl.max_blocks_per_seq * 16 + 1
    out = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(out[0]).all() and np.isfinite(out[1]).all()
    d["context_lens"][0] = -1
    out = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(out[0]).all()


def test_split_length_beyond_workspace_flags_bounds(pf):
    wl = make_workload("badsplit", 2, 4, 2, 64, 16, [100, 300], seed=53)
    d = to_device(wl)
    ws = pf.alloc_workspace(2, 4, 64, 200, 64, "cuda")
    pf.paged_attention_decode_partition(*attn_args(d), 64, 200, ws)
    out = pf.paged_attention_merge(ws, d["context_lens"], 4, 64, 64, 200).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isfinite(out[0]).all() and np.isnan(out[1]).all()


def test_split_bad_block_id_flags_bounds(pf, oracle_lib):
    """The persistent partition pass meets a table entry outside the pool: that partition's
    partial is NaN, the merge carries it into the sequence's rows, and the word is set."""
    wl = make_workload("badblks", 3, 8, 2, 128, 16, [40, 50, 60], seed=54, pool_scale=2)
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    d = to_device(wl)
    d["block_tables"][1, 2] = wl.num_blocks            # seq 1, tokens 32..47
    ws = pf.alloc_workspace(3, 8, 128, 64, 32, "cuda")
    pf.paged_attention_decode_partition(*attn_args(d), 32, 64, ws)
    out = pf.paged_attention_merge(ws, d["context_lens"], 8, 128, 32, 64).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(out[1]).all()
    check_close(out[[0, 2]], ref[[0, 2]])


def test_bounded_wait_times_out_and_context_survives(pf):
    torch.cuda.synchronize()
    assert pf.get_device_error() == pf.PF_OK
    pf.debug_bounded_wait(50_000_000)                  # 50 ms, then give up
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_TIMEOUT
    assert pf.get_device_error() == pf.PF_OK
    x = torch.ones(1024, device="cuda")                # the context is still usable
    assert float(x.sum()) == 1024.0


def test_host_argument_errors(pf):
    wl = make_workload("args", 2, 4, 2, 64, 16, [10, 20], seed=54)
    d = to_device(wl)
    q, kc, vc, bt, cl = attn_args(d)
    L = pf.lib()
    cases = [
        (dict(num_seqs=-1), pf.PF_ERR_INVALID_ARG),
        (dict(num_q_heads=3), pf.PF_ERR_INVALID_ARG),          # not a multiple of num_kv_heads
        (dict(head_dim=96), pf.PF_ERR_UNSUPPORTED),
        (dict(block_size=8), pf.PF_ERR_UNSUPPORTED),
        (dict(num_q_heads=32), pf.PF_ERR_UNSUPPORTED),         # group 16
        (dict(scale=float("nan")), pf.PF_ERR_INVALID_ARG),
        (dict(q=q.data_ptr() + 2), pf.PF_ERR_INVALID_ARG),     # misaligned
        (dict(num_blocks=0), pf.PF_ERR_INVALID_ARG),
    ]
    out = torch.empty((2, 4, 64), dtype=torch.float32, device="cuda")
    for change, want in cases:
        a = dict(q=q.data_ptr(), kc=kc.data_ptr(), vc=vc.data_ptr(), bt=bt.data_ptr(), cl=cl.data_ptr(),
                 num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                 mb=wl.max_blocks_per_seq, num_blocks=wl.num_blocks, scale=0.125)
        a.update(change)
        st = L.pf_paged_attention_decode(a["q"], a["kc"], a["vc"], a["bt"], a["cl"], a["num_seqs"],
                                         a["num_q_heads"], a["num_kv_heads"], a["head_dim"], a["block_size"],
                                         a["mb"], a["num_blocks"], a["scale"], out.data_ptr(), None)
        assert st == want, (change, st)
    with pytest.raises(TypeError):
        pf.paged_attention_decode(q.float(), kc, vc, bt, cl)
    with pytest.raises(ValueError):
        pf.paged_attention_decode(q.cpu(), kc, vc, bt, cl)
