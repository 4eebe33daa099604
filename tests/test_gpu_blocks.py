"""Block copy (pf_copy_blocks) on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from tests.helpers import attn_args, bits, to_device
from workloads import make_workload

pytestmark = pytest.mark.gpu


def _pairs(wl, n, seed):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(wl.num_blocks)
    return np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)   # distinct, no dst is a src


@pytest.mark.parametrize("Hkv,D,bs", [(8, 128, 16), (2, 64, 32), (3, 72, 7), (32, 128, 16), (1, 8, 1)])
def test_copy_blocks_bit_exact(pf, oracle_lib, Hkv, D, bs):
    wl = make_workload("copy", 3, Hkv, Hkv, D, bs, [40, 17, 64], seed=Hkv + D + bs, pool_scale=4)
    pairs = _pairs(wl, max(1, wl.num_blocks // 3), seed=D)
    d = to_device(wl)
    pf.copy_blocks(d["k_cache"], d["v_cache"], torch.from_numpy(pairs).cuda())
    assert pf.get_device_error() == pf.PF_OK
    ek, ev, bad = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, pairs)
    assert bad == 0
    assert np.array_equal(bits(d["k_cache"]), ek) and np.array_equal(bits(d["v_cache"]), ev)


def test_copy_blocks_out_of_range_and_identity(pf, oracle_lib):
    wl = make_workload("copy", 2, 4, 4, 64, 16, [30, 50], seed=71, pool_scale=4)
    pairs = _pairs(wl, 3, seed=1)
    mapping = np.concatenate([pairs, [[-1, pairs[0, 1]], [pairs[1, 0], wl.num_blocks], [2, 2]]])
    d = to_device(wl)
    pf.copy_blocks(d["k_cache"], d["v_cache"], torch.from_numpy(mapping).cuda())
    assert pf.get_device_error() == pf.PF_ERR_DEVICE_BOUNDS
    ek, ev, bad = oracle_lib.copy_blocks(wl.k_cache, wl.v_cache, mapping)
    assert bad == 2
    assert np.array_equal(bits(d["k_cache"]), ek) and np.array_equal(bits(d["v_cache"]), ev)


def test_forked_sequence_decodes_like_its_parent(pf):
    wl = make_workload("fork", 3, 8, 2, 128, 16, [45, 70, 33], seed=72, pool_scale=2)
    d = to_device(wl)
    parent = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    i = 1
    nb = int((wl.context_lens[i] + 15) // 16)
    fresh = int(np.setdiff1d(np.arange(wl.num_blocks), wl.block_tables[wl.block_tables >= 0])[0])
    pf.copy_blocks(d["k_cache"], d["v_cache"], torch.tensor([[int(wl.block_tables[i, nb - 1]), fresh]],
                                                            dtype=torch.int64, device="cuda"))
    d["block_tables"][i, nb - 1] = fresh
    child = pf.paged_attention_decode(*attn_args(d)).cpu().numpy()
    assert pf.get_device_error() == pf.PF_OK
    assert np.array_equal(child, parent)


def test_copy_blocks_full_size(pf):
    """4096 pairs of Llama-3-8B-shaped blocks (8 kv heads x 16 x 128): 268 MB each way,
    the launch the bench times, checked against torch indexing."""
    NB, shape = 8192, (8, 16, 128)
    g = torch.Generator(device="cuda").manual_seed(5)
    kc = torch.randint(-32768, 32767, (NB,) + shape, dtype=torch.int16, device="cuda", generator=g)
    vc = torch.randint(-32768, 32767, (NB,) + shape, dtype=torch.int16, device="cuda", generator=g)
    perm = torch.randperm(NB, device="cuda", generator=g)
    mapping = torch.stack([perm[:4096], perm[4096:]], dim=1).contiguous()
    k0, v0 = kc.clone(), vc.clone()
    pf.copy_blocks(kc, vc, mapping)
    assert pf.get_device_error() == pf.PF_OK
    ek, ev = k0.clone(), v0.clone()
    ek[mapping[:, 1]] = k0[mapping[:, 0]]
    ev[mapping[:, 1]] = v0[mapping[:, 0]]
    assert torch.equal(kc, ek) and torch.equal(vc, ev)
