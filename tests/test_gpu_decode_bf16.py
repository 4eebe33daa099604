"""Single-pass decode with a bf16 output (pf_paged_attention_decode_bf16).

Two checks: against the fp64 oracle with the bf16 output's bound |d| <= 2e-3 + 1e-2 |ref|
(the fp32 error plus one bf16 rounding, a relative 2^-9), and bit for bit against the fp32
entry's output rounded to bf16 (nearest, ties to even) on the host -- the two entry points run
the same arithmetic and differ only in that last rounding.
"""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, to_device
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, make_workload

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_bf16_close(got_bits, ref):
    got = bf16_bits_to_f32(got_bits).astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    d = np.abs(got - ref)
    bound = 2e-3 + 1e-2 * np.abs(ref)
    worst = float((d - bound).max()) if d.size else 0.0
    assert worst <= 0.0, (float(d.max()), worst)


def run_both(pf, d):
    b = pf.paged_attention_decode_bf16(*attn_args(d))
    assert pf.get_device_error() == pf.PF_OK
    f = pf.paged_attention_decode(*attn_args(d))
    assert pf.get_device_error() == pf.PF_OK
    assert b.dtype == torch.bfloat16 and b.shape == f.shape
    return _bits(b), f.cpu().numpy()


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_named_workloads_against_oracle_and_fp32(pf, oracle_lib, config_workload, index):
    """Every output of the five named workloads (the Llama-3-shaped one at full size; the
    continuous-batch one after its append, as its step runs)."""
    wl = config_workload(index)
    d = to_device(wl)
    kc, vc = wl.k_cache, wl.v_cache
    if wl.slot_mapping is not None:
        pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
        kc, vc, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, kc, vc, wl.block_size)
    bits, f32 = run_both(pf, d)
    assert np.array_equal(bits, f32_to_bf16_bits(f32))
    ref = oracle_lib.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    check_bf16_close(bits, ref)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_every_group_and_head_dim(pf, oracle_lib, D, g):
    lengths = [0, 1, 15, 16, 17, 300, 1000]
    wl = make_workload("bf16", len(lengths), 8 * g, 8, D, 16, lengths, seed=200 + g + D, pool_scale=2)
    bits, f32 = run_both(pf, to_device(wl))
    assert np.array_equal(bits, f32_to_bf16_bits(f32))
    assert not bits[0].any()  # an empty sequence gives +0.0 everywhere
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_bf16_close(bits, ref)


def test_bad_block_gives_nan_rows(pf, oracle_lib):
    wl = make_workload("bf16bad", 3, 16, 4, 128, 16, [200, 300, 100], seed=210, pool_scale=2)
    d = to_device(wl)
    d["block_tables"][1, 4] = wl.num_blocks + 1
    out = pf.paged_attention_decode_bf16(*attn_args(d))
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    got = bf16_bits_to_f32(_bits(out))
    assert np.isnan(got[1]).all()
    ref = oracle_lib.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale)
    check_bf16_close(_bits(out)[[0, 2]], ref[[0, 2]])


def test_int16_view_output_and_repeats(pf):
    """The output may be given as an int16 view of bf16 bits; repeated calls are bit-identical."""
    wl = make_workload("bf16rep", 6, 32, 8, 128, 16, ("uniform", 1, 3000), seed=211, pool_scale=2)
    d = to_device(wl)
    out = torch.empty((6, 32, 128), dtype=torch.int16, device="cuda")
    first = pf.paged_attention_decode_bf16(*attn_args(d), out=out).clone()
    for _ in range(20):
        assert torch.equal(pf.paged_attention_decode_bf16(*attn_args(d), out=out), first)
    assert pf.get_device_error() == pf.PF_OK
