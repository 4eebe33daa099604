"""Fused append + decode (pf_paged_attention_decode_append) on the GPU.

Its definition is the two-step sequence append-then-attend; it is checked against
the oracle's append and attention (caches bit-exact, output within tolerance) and
against the library's own two launches (bit-identical)."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, bits, check_close, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def fused(pf, d):
    out = pf.paged_attention_decode_append(d["q"], d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"],
                                           d["v_cache"], d["block_tables"], d["context_lens"])
    return out


def two_step(pf, d):
    pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    return pf.paged_attention_decode(*attn_args(d))


def oracle_step(orc, wl, slots=None):
    slots = wl.slot_mapping if slots is None else slots
    kc, vc, _ = orc.reshape_and_cache(wl.new_k, wl.new_v, slots, wl.k_cache, wl.v_cache, wl.block_size)
    return kc, vc, orc.paged_attention(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)


def test_cont_batch_fused_step(pf, oracle_lib, config_workload):
    wl = config_workload(3)
    d = to_device(wl)
    out = fused(pf, d).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    kc, vc, ref = oracle_step(oracle_lib, wl)
    assert np.array_equal(bits(d["k_cache"]), kc) and np.array_equal(bits(d["v_cache"]), vc)
    check_close(out, ref)
    d2 = to_device(wl)
    out2 = two_step(pf, d2).cpu().numpy()
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_fused_step_shapes(pf, oracle_lib, D, g, bs):
    lengths = [1, 15, 16, 17, 33, 100, 512, 513]
    wl = make_workload("fa", len(lengths), 2 * g, 2, D, bs, lengths, seed=D + g + bs, pool_scale=2, append=True,
                       num_skip_slots=2)
    d = to_device(wl)
    out = fused(pf, d).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    kc, vc, ref = oracle_step(oracle_lib, wl)
    assert np.array_equal(bits(d["k_cache"]), kc) and np.array_equal(bits(d["v_cache"]), vc)
    check_close(out, ref)


def test_slot_that_is_not_the_newest_position_is_rejected(pf, oracle_lib):
    wl = make_workload("fa", 3, 8, 2, 128, 16, [20, 40, 33], seed=81, pool_scale=2, append=True)
    slots = wl.slot_mapping.copy()
    slots[1] = slots[1] - 1                      # one position too early
    d = to_device(wl)
    d["slot_mapping"] = torch.from_numpy(slots).cuda()
    out = fused(pf, d).cpu().numpy()
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert np.isnan(out[1]).all()
    good = slots.copy()
    good[1] = -1                                 # sequence 1 must have written nothing
    kc, vc, ref = oracle_step(oracle_lib, wl, good)
    assert np.array_equal(bits(d["k_cache"]), kc) and np.array_equal(bits(d["v_cache"]), vc)
    check_close(out[[0, 2]], ref[[0, 2]])
