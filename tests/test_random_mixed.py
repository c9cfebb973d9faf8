"""Randomized continuous batches against the oracle.

Each seed draws a batch that mixes what the named configurations keep apart:
- 1 to 8 kv heads and 1 to 16 query heads per kv head;
- 1 to 24 sequences, each a decode row (60 %), a short speculative chunk of
  2-8 rows (15 %) or a prefill chunk of 9-599 rows (25 %);
- 0 to 8000 cached tokens before the new ones;
- a quarter of the batches with a shared prefix of 1-64 pages (cascade);
- a third on FP8 pages.

Every call runs twice and must give the same bits; up to 256 sampled rows (all
rows of smaller batches) are checked against the float64 oracle within
max |err| 1e-2, mean 1e-3.  The oracle's work is bounded by shortening the
cached contexts of the largest draws.
"""

import numpy as np
import pytest
import torch

import oracle.pkv_oracle as O
import paged_kv_cache_pkv_gb300 as pkv
from helpers import bits, compare, oracle_attend, oracle_write, to_device
from workloads import fp8_pools, make_batch

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng(7000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    while G * hkv > 64:
        G //= 2
    B = int(rng.integers(1, 25))
    kinds = rng.choice(["decode", "spec", "chunk"], size=B, p=[0.6, 0.15, 0.25])
    q = np.where(kinds == "decode", 1,
                 np.where(kinds == "spec", rng.integers(2, 9, B), rng.integers(9, 600, B)))
    prefix = 16 * int(rng.integers(1, 65)) if rng.random() < 0.25 else 0
    L = q + rng.integers(0, 8000, B)
    if prefix:  # no new token in the shared pages, and every row sees a key of its own
        L = np.maximum(L, q + prefix)
    fp8 = bool(rng.random() < 0.35)
    while int((q * G * hkv * L).sum()) > 6e8:
        L = np.maximum(q + prefix, L // 2)
    return G * hkv, hkv, q, L, prefix, fp8


@pytest.mark.parametrize("seed", range(30))
def test_random_mixed_batch(pkvlib, seed):
    hq, hkv, q, L, prefix, fp8 = _draw(seed)
    what = f"seed {seed}: B={len(q)} hq/hkv={hq}/{hkv} fp8={fp8} prefix={prefix}"
    b = make_batch(L.tolist(), q.tolist(), hq, hkv, seed=8000 + seed, device="cuda",
                   shared_prefix_tokens=prefix)
    meta = to_device(b)
    T = int(b.query_start_loc[-1])
    rows = None if T <= 256 else sorted(np.random.default_rng(seed).choice(T, 256, replace=False).tolist())
    kw = dict(max_query_len=int(q.max()), shared_prefix_pages=prefix // 16)
    if fp8:
        pools = fp8_pools(b, 9000 + seed)
        kc, vc, ks, vs = (t.clone() for t in pools)
        pkv.write_fp8(b.k_new, b.v_new, meta["slot_mapping"], kc, vc, ks, vs)
        run = lambda: pkv.attend_fp8(b.q, kc, vc, ks, vs, meta["block_tables"], meta["seq_lens"],
                                     meta["query_start_loc"], b.scale, **kw)
    else:
        kc, vc = b.k_cache.clone(), b.v_cache.clone()
        pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
        run = lambda: pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"],
                                 meta["query_start_loc"], b.scale, **kw)
    first = run().clone()
    second = run().clone()
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0, what
    assert torch.equal(first, second), f"{what}: two calls differ"
    if fp8:
        u8 = lambda t: t.detach().contiguous().cpu().numpy()
        ref = O.write_fp8(bits(b.k_new), bits(b.v_new), b.slot_mapping, *(u8(t) for t in pools), b.page_size)
        expected = O.attend_fp8(bits(b.q), *ref, b.block_tables, b.seq_lens, b.query_start_loc, b.scale,
                                b.num_q_heads, b.num_kv_heads, b.page_size, rows=rows)
    else:
        k_ref, v_ref = oracle_write(b)
        expected = oracle_attend(b, k_ref, v_ref, rows=rows)
    compare(first, expected, rows=rows, what=what)
