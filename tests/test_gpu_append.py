"""KV append (pf_reshape_and_cache) on the GPU: bit-exact against the oracle's scatter."""
import numpy as np
import pytest
import torch

from tests.helpers import bits, numpy_scatter, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def test_cont_batch_append_bit_exact(pf, oracle_lib, config_workload):
    wl = config_workload(3)           # 64 new tokens, 8 of them with slot -1
    d = to_device(wl)
    pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    assert pf.get_device_error() == pf.PF_OK
    ok, ov, bad = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache,
                                               wl.block_size)
    assert bad == 0
    assert np.array_equal(bits(d["k_cache"]), ok)
    assert np.array_equal(bits(d["v_cache"]), ov)


@pytest.mark.parametrize("Hkv,D,bs", [(1, 8, 1), (2, 64, 16), (8, 128, 32), (3, 72, 7), (32, 128, 16)])
def test_append_shapes_sentinel_and_skip(pf, oracle_lib, Hkv, D, bs):
    wl = make_workload("app", 6, Hkv, Hkv, D, bs, [5, 1, 40, 17, 33, 2], seed=D + bs, pool_scale=2, append=True,
                       num_skip_slots=2)
    # sentinel caches: every slot not written must keep its bits
    wl.k_cache = np.full_like(wl.k_cache, 0x3F80)          # 1.0
    wl.v_cache = np.full_like(wl.v_cache, 0xBF80)          # -1.0
    d = to_device(wl)
    pf.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    assert pf.get_device_error() == pf.PF_OK
    ek, ev, _ = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, wl.slot_mapping, wl.k_cache, wl.v_cache, bs)
    assert np.array_equal(bits(d["k_cache"]), ek) and np.array_equal(bits(d["v_cache"]), ev)
    nk, nv = numpy_scatter(wl)
    assert np.array_equal(ek, nk) and np.array_equal(ev, nv)
    assert (wl.slot_mapping == -1).sum() >= 2


def test_out_of_range_slots_are_skipped_and_reported(pf, oracle_lib):
    wl = make_workload("app", 4, 2, 2, 64, 16, [4, 17, 30, 2], seed=21, pool_scale=2, append=True)
    slots = wl.slot_mapping.copy()
    slots[1] = -5
    slots[2] = wl.num_blocks * wl.block_size
    d = to_device(wl)
    sm = torch.from_numpy(slots).cuda()
    pf.reshape_and_cache(d["new_k"], d["new_v"], sm, d["k_cache"], d["v_cache"])
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    assert pf.get_device_error() == pf.PF_OK               # reading clears the word
    ek, ev, bad = oracle_lib.reshape_and_cache(wl.new_k, wl.new_v, slots, wl.k_cache, wl.v_cache, 16)
    assert bad == 2
    assert np.array_equal(bits(d["k_cache"]), ek) and np.array_equal(bits(d["v_cache"]), ev)


def test_zero_tokens_is_a_no_op(pf):
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    empty = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    pf.reshape_and_cache(empty, empty, torch.zeros(0, dtype=torch.int64, device="cuda"), kc, vc)
    assert pf.get_device_error() == pf.PF_OK
    assert not kc.any() and not vc.any()
