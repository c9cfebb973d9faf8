"""pkv_write parity: bit-exact against the oracle's write, pool canaries intact."""

import numpy as np
import pytest
import torch

import paged_kv_cache_pkv_gb300 as pkv
from helpers import bits, oracle_write, to_device
from workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def _run_write(batch, slots=None):
    meta = to_device(batch)
    if slots is not None:
        meta["slot_mapping"] = torch.from_numpy(np.asarray(slots, np.int64)).cuda()
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    pkv.write(batch.k_new, batch.v_new, meta["slot_mapping"], kc, vc)
    torch.cuda.synchronize()
    return kc, vc


@pytest.mark.parametrize("idx", [1, 2, 4, 5])
def test_write_bit_exact_named(pkvlib, idx):
    b = workload(idx, device="cuda")
    kc, vc = _run_write(b)
    k_ref, v_ref = oracle_write(b)
    assert np.array_equal(bits(kc), k_ref)
    assert np.array_equal(bits(vc), v_ref)
    assert pkv.get_last_error() == 0


def test_write_bit_exact_long_tail_pages(pkvlib):
    """Config 3 (4.5 GB of pool): written pages compared on the host, every
    other page compared with the untouched pool on the device."""
    b = workload(3, device="cuda")
    kc, vc = _run_write(b)
    pages = np.unique(b.slot_mapping // b.page_size)
    k_new, v_new = bits(b.k_new), bits(b.v_new)
    small_k = bits(b.k_cache[torch.from_numpy(pages).cuda()])
    small_v = bits(b.v_cache[torch.from_numpy(pages).cuda()])
    # the oracle write restricted to the touched pages, renumbered
    remap = {int(p): i for i, p in enumerate(pages)}
    slots_small = np.array([remap[int(s) // 16] * 16 + int(s) % 16 for s in b.slot_mapping])
    import oracle.pkv_oracle as O
    k_ref, v_ref = O.write(k_new, v_new, slots_small, small_k, small_v, 16)
    idx = torch.from_numpy(pages).cuda()
    assert np.array_equal(bits(kc[idx]), k_ref)
    assert np.array_equal(bits(vc[idx]), v_ref)
    keep = torch.ones(b.num_blocks, dtype=torch.bool, device="cuda")
    keep[idx] = False
    assert torch.equal(kc[keep].view(torch.int16), b.k_cache[keep].view(torch.int16))
    assert torch.equal(vc[keep].view(torch.int16), b.v_cache[keep].view(torch.int16))


def test_write_padding_and_ragged(pkvlib):
    b = make_batch([5, 33, 16, 40, 129], [2, 1, 16, 3, 77], 4, 2, seed=5, device="cuda")
    slots = b.slot_mapping.copy()
    slots[[0, 5, 20]] = -1
    kc, vc = _run_write(b, slots)
    k_ref, v_ref = oracle_write(b, slots)
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)


def test_write_slot_beyond_pool_is_flagged_and_skipped(pkvlib):
    b = make_batch([20, 7], [3, 2], 8, 8, seed=6, device="cuda")
    pkv.get_last_error()  # clear
    slots = b.slot_mapping.copy()
    slots[1] = b.num_blocks * 16 + 5  # outside the pool
    kc, vc = _run_write(b, slots)
    assert pkv.get_last_error() & pkv.STATUS_BAD_SLOT
    slots_ok = slots.copy()
    slots_ok[1] = -1
    k_ref, v_ref = oracle_write(b, slots_ok)
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)
    assert pkv.get_last_error() == 0  # cleared by the read


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 2), (16, 1)])
def test_write_head_counts(pkvlib, hq, hkv):
    b = make_batch([50, 3, 300], [50, 1, 17], hq, hkv, seed=7, device="cuda")
    kc, vc = _run_write(b)
    k_ref, v_ref = oracle_write(b)
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)
