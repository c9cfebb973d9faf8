"""Page pool: allocation, reference counts of shared pages, usage gauge
(host side, no GPU), and the copy-on-write page copy (GPU)."""

import random

import numpy as np
import pytest
import torch

import paged_kv_cache_pkv_gb300 as pkv
from helpers import bits
from workloads import make_batch


def test_alloc_release_and_usage(pkvlib):
    pool = pkv.PagePool(10)
    a = pool.alloc(4)
    assert len(set(a)) == 4 and all(0 <= x < 10 for x in a)
    assert pool.usage() == (4, 10)
    b = pool.alloc(6)
    assert pool.usage() == (10, 10) and not set(a) & set(b)
    with pytest.raises(pkv.PkvError) as e:
        pool.alloc(1)
    assert e.value.code == -10
    pool.release(a[:2])
    assert pool.usage() == (8, 10)
    c = pool.alloc(2)
    assert set(c) == set(a[:2])  # freed pages come back first
    pool.close()


def test_shared_prefix_pages_are_freed_by_the_last_user(pkvlib):
    pool = pkv.PagePool(8)
    prefix = pool.alloc(3)
    pool.retain(prefix)  # a second sequence reuses the prefix
    assert [pool.refcount(x) for x in prefix] == [2, 2, 2]
    pool.release(prefix)
    assert pool.usage() == (3, 8)
    pool.release(prefix)
    assert pool.usage() == (0, 8)


def test_bad_releases_change_nothing(pkvlib):
    pool = pkv.PagePool(6)
    a = pool.alloc(2)
    for bad, code in (([a[0], 5], -8), ([a[0], a[0]], -8), ([7], -4), ([-1], -4)):
        with pytest.raises(pkv.PkvError) as e:
            pool.release(bad)
        assert e.value.code == code
        assert pool.usage() == (2, 6) and pool.refcount(a[0]) == 1
    with pytest.raises(pkv.PkvError):
        pool.retain([4])  # not allocated


def test_random_operations_match_a_model(pkvlib):
    rng = random.Random(0)
    pool, refs = pkv.PagePool(64), {}
    for _ in range(3000):
        op = rng.random()
        live = [p for p, r in refs.items() if r > 0]
        if op < 0.4:
            n = rng.randint(0, 8)
            free = 64 - len(live)
            if n > free:
                with pytest.raises(pkv.PkvError):
                    pool.alloc(n)
            else:
                got = pool.alloc(n)
                assert not set(got) & set(live)
                for p in got:
                    refs[p] = 1
        elif op < 0.6 and live:
            pick = rng.sample(live, rng.randint(1, min(4, len(live))))
            pool.retain(pick)
            for p in pick:
                refs[p] += 1
        elif live:
            pick = rng.sample(live, rng.randint(1, min(4, len(live))))
            pool.release(pick)
            for p in pick:
                refs[p] -= 1
        used = sum(1 for r in refs.values() if r > 0)
        assert pool.usage() == (used, 64)
    for p, r in refs.items():
        assert pool.refcount(p) == r


@pytest.mark.gpu
def test_copy_on_write_of_a_shared_last_page(pkvlib):
    """Two sequences share a partly filled page; the one that appends gets a
    private copy of the written rows and the other keeps the original."""
    b = make_batch([40], [1], 8, 2, seed=3, device="cuda", pool_factor=3.0)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pool = pkv.PagePool(b.num_blocks)
    pages = pool.alloc(3)
    pool.retain(pages[2:])  # the last page (rows 0..7 written) is shared
    k_before, v_before = bits(kc), bits(vc)
    new = pool.make_writable(pages[2], 8, kc, vc)
    torch.cuda.synchronize()
    assert new != pages[2] and pool.refcount(pages[2]) == 1 and pool.refcount(new) == 1
    k_after, v_after = bits(kc), bits(vc)
    assert np.array_equal(k_after[new, :, :8], k_before[pages[2], :, :8])
    assert np.array_equal(v_after[new, :, :8], v_before[pages[2], :, :8])
    keep = np.ones(b.num_blocks, bool)
    keep[new] = False
    assert np.array_equal(k_after[keep], k_before[keep]) and np.array_equal(v_after[keep], v_before[keep])
    assert np.array_equal(k_after[new, :, 8:], k_before[new, :, 8:])  # rows past the copy untouched
    # a private page is returned as is
    assert pool.make_writable(new, 8, kc, vc) == new
    pool.close()


def test_oracle_export_import_roundtrip():
    rng = np.random.default_rng(0)
    kc = rng.integers(0, 2 ** 16, size=(7, 2, 16, 128), dtype=np.uint64).astype(np.uint16)
    vc = rng.integers(0, 2 ** 16, size=(7, 2, 16, 128), dtype=np.uint64).astype(np.uint16)
    import oracle.pkv_oracle as O
    buf = O.export_pages(kc, vc, [5, 1, 3])
    assert buf.shape == (3, 2, 2, 16, 128)
    assert np.array_equal(buf[0, 0], kc[5]) and np.array_equal(buf[2, 1], vc[3])
    k2, v2 = O.import_pages(buf, [0, 2, 4], np.zeros_like(kc), np.zeros_like(vc))
    assert np.array_equal(k2[2], kc[1]) and np.array_equal(v2[4], vc[3]) and not k2[1].any()


@pytest.mark.gpu
@pytest.mark.parametrize("host_buffer", [False, True])
def test_export_import_pages_bit_exact(pkvlib, host_buffer):
    import oracle.pkv_oracle as O
    b = make_batch([300, 40], [1, 1], 32, 8, seed=4, device="cuda", pool_factor=1.5)
    pages = np.array([int(x) for x in b.block_tables[0, :19]] + [int(b.block_tables[1, 2])], dtype=np.int32)
    pt = torch.from_numpy(pages).cuda()
    out = torch.empty((len(pages), 2, 8, 16, 128), dtype=torch.bfloat16,
                      pin_memory=True) if host_buffer else None
    buf = pkv.export_pages(b.k_cache, b.v_cache, pt, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(buf), O.export_pages(bits(b.k_cache), bits(b.v_cache), pages))
    # import into a fresh pool at other pages
    kc2, vc2 = torch.zeros_like(b.k_cache), torch.zeros_like(b.v_cache)
    dst = np.arange(len(pages), dtype=np.int32)[::-1].copy() + 3
    pkv.import_pages(buf, torch.from_numpy(dst).cuda(), kc2, vc2)
    torch.cuda.synchronize()
    k_ref, v_ref = O.import_pages(bits(buf), dst, bits(kc2 * 0), bits(vc2 * 0))
    assert np.array_equal(bits(kc2), k_ref) and np.array_equal(bits(vc2), v_ref)
    assert pkv.get_last_error() == 0
