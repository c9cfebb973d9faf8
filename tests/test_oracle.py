"""Pins for the float64 oracle: checks against things other than itself.

Each check is a function of the oracle module so that the same check can be
run against deliberately broken copies of the oracle (planted mistakes, at the
bottom of this file): a plausible slip anywhere in the oracle -- a wrong
kv-head mapping, top-left instead of bottom-right causal alignment, a missing
scale, the page/row split swapped -- must fail at least one pin.
"""

import math
import types

import numpy as np
import pytest
import torch

import oracle.pkv_oracle as O
from workloads import make_batch, workload


def _bits(x_f32: torch.Tensor) -> np.ndarray:
    return x_f32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_bits(rng, shape, scale=1.0):
    return _bits(torch.from_numpy((scale * rng.standard_normal(shape)).astype(np.float32)))


def _pool_from_contiguous(K_bits, perm, P):
    """Place a contiguous [L, Hkv, D] sequence into a pool at pages ``perm``."""
    L, Hkv, D = K_bits.shape
    npages = (L + P - 1) // P
    NB = int(max(perm[:npages])) + 3
    pool = np.full((NB, Hkv, P, D), 0x7FC0, dtype=np.uint16)  # NaN filler
    for j in range(L):
        pool[perm[j // P], :, j % P, :] = K_bits[j]
    return pool


# --------------------------------------------------------------------------
# bf16 widening: pinned to torch's own bf16 -> float64 conversion and to
# hand-known bit patterns.
# --------------------------------------------------------------------------

def test_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F80, 0x0000, 0x8000], dtype=np.uint16)
    got = O.bf16_to_f64(bits)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, math.inf, 0.0, -0.0]
    assert list(got) == want
    assert math.copysign(1.0, got[-1]) == -1.0


def test_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 16, size=4096, dtype=np.uint64).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # skip inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_to_f64(bits), ref)


# --------------------------------------------------------------------------
# write: every written row is found again by gathering through the block
# table at its logical position; everything else is untouched.
# --------------------------------------------------------------------------

def check_write_roundtrip(orc):
    b = make_batch([5, 33, 16, 40], [2, 1, 16, 3], 4, 2, seed=11, pool_factor=2.0)
    k_new, v_new = b.k_new.view(torch.int16).numpy().view(np.uint16), b.v_new.view(torch.int16).numpy().view(np.uint16)
    kc = b.k_cache.view(torch.int16).numpy().view(np.uint16)
    vc = b.v_cache.view(torch.int16).numpy().view(np.uint16)
    slots = b.slot_mapping.copy()
    slots[1] = -1  # padding token: must not be written
    k2, v2 = orc.write(k_new, v_new, slots, kc, vc, b.page_size)
    ok = True
    touched = np.zeros(kc.shape[:1] + kc.shape[2:3], dtype=bool)  # [NB, P]
    for bi in range(b.B):
        L, n = int(b.seq_lens[bi]), int(b.q_lens[bi])
        Kg = orc.gather(k2, b.block_tables[bi], L, b.page_size)
        Vg = orc.gather(v2, b.block_tables[bi], L, b.page_size)
        for j in range(n):
            t = int(b.query_start_loc[bi]) + j
            if slots[t] < 0:
                continue
            touched[slots[t] // b.page_size, slots[t] % b.page_size] = True
            ok &= np.array_equal(Kg[L - n + j], O.bf16_to_f64(k_new[t]))
            ok &= np.array_equal(Vg[L - n + j], O.bf16_to_f64(v_new[t]))
    # canaries: every other (page, row) keeps its old bits, including the
    # padding token's slot
    mask = ~touched[:, None, :, None]
    ok &= np.array_equal(np.where(mask, k2, 0), np.where(mask, kc, 0))
    ok &= np.array_equal(np.where(mask, v2, 0), np.where(mask, vc, 0))
    return bool(ok)


def test_write_roundtrip():
    assert check_write_roundtrip(O)


def test_write_does_not_modify_inputs_and_rejects_outside_pool():
    kc = np.zeros((2, 1, 4, 3), dtype=np.uint16)
    new = np.ones((1, 1, 3), dtype=np.uint16)
    O.write(new, new, np.array([5]), kc, kc, 4)
    assert not kc.any()
    with pytest.raises(IndexError):
        O.write(new, new, np.array([8]), kc, kc, 4)


# --------------------------------------------------------------------------
# paging: the result does not depend on where pages live in the pool
# (bit-identical, since the gathered float64 arrays are identical).
# --------------------------------------------------------------------------

def check_paged_equals_contiguous(orc):
    rng = np.random.default_rng(3)
    P, Hkv, Hq, D, L = 4, 2, 4, 8, 23
    K = _rand_bits(rng, (L, Hkv, D))
    V = _rand_bits(rng, (L, Hkv, D))
    q = _rand_bits(rng, (3, Hq, D))
    npages = (L + P - 1) // P
    outs = []
    for trial in range(4):
        perm = np.arange(npages) if trial == 0 else rng.permutation(npages + 5)[:npages]
        kp = _pool_from_contiguous(K, perm, P)
        vp = _pool_from_contiguous(V, perm, P)
        bt = np.asarray(perm, dtype=np.int32)[None, :]
        outs.append(orc.attend(q, kp, vp, bt, np.array([L]), np.array([0, 3]), 0.3, Hq, Hkv, P))
    # the contiguous case: a single "page" holding the whole sequence
    kp1 = K.transpose(1, 0, 2)[None]
    vp1 = V.transpose(1, 0, 2)[None]
    outs.append(orc.attend(q, kp1, vp1, np.zeros((1, 1), np.int32), np.array([L]),
                           np.array([0, 3]), 0.3, Hq, Hkv, L))
    return all(np.array_equal(outs[0], o) for o in outs[1:])


def test_paged_equals_contiguous():
    assert check_paged_equals_contiguous(O)


# --------------------------------------------------------------------------
# closed forms of softmax attention
# --------------------------------------------------------------------------

def test_softmax_of_small_integers():
    """Scores 0, 1, 2 with one-hot values: out = softmax([0, 1, 2])."""
    D = 4
    q = np.zeros(D); q[0] = 1.0
    keys = np.zeros((3, D)); keys[:, 0] = [0.0, 1.0, 2.0]
    values = np.eye(3, D)
    out = O.attend_one(q, keys, values, 1.0)
    z = 1.0 + math.e + math.e ** 2
    assert np.allclose(out[:3], [1 / z, math.e / z, math.e ** 2 / z], rtol=0, atol=1e-15)
    assert out[3] == 0.0


def test_constant_values_return_that_value():
    rng = np.random.default_rng(1)
    keys = rng.standard_normal((37, 16))
    v = rng.standard_normal(16)
    out = O.attend_one(rng.standard_normal(16), keys, np.tile(v, (37, 1)), 0.25)
    assert np.allclose(out, v, rtol=0, atol=1e-13)


def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((1, 8))
    out = O.attend_one(rng.standard_normal(8), rng.standard_normal((1, 8)), v, 1.7)
    assert np.array_equal(out, v[0])


def test_weights_are_a_probability_vector_with_exponential_ratios():
    rng = np.random.default_rng(4)
    n, D = 9, 16
    q, keys = rng.standard_normal(D), rng.standard_normal((n, D))
    w = O.attend_one(q, keys, np.eye(n, D), 0.5)[:n]
    assert abs(w.sum() - 1.0) < 1e-12 and (w > 0).all()
    s = 0.5 * keys @ q
    for a in range(n):
        for c in range(n):
            assert abs(math.log(w[a] / w[c]) - (s[a] - s[c])) < 1e-12


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(5)
    keys, values = rng.standard_normal((21, 8)), rng.standard_normal((21, 8))
    out = O.attend_one(np.zeros(8), keys, values, 0.9)
    assert np.allclose(out, values.mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(6)
    D = 128
    q = rng.standard_normal(D)
    keys = rng.standard_normal((50, D)) * 0.01
    keys[17] = 40.0 * q / np.linalg.norm(q) * math.sqrt(D)
    values = rng.standard_normal((50, D))
    out = O.attend_one(q, keys, values, 1.0 / math.sqrt(D))
    assert np.allclose(out, values[17], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# library special cases: torch scaled_dot_product_attention in float64
# --------------------------------------------------------------------------

def _sdpa(q, k, v, scale, causal):
    # q: [n, Hq, D], k/v: [L, Hq, D] float64 -> [n, Hq, D]
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1), torch.from_numpy(k).transpose(0, 1),
        torch.from_numpy(v).transpose(0, 1), is_causal=causal, scale=scale)
    return out.transpose(0, 1).numpy()


def check_matches_sdpa(orc, Hq, Hkv, L, n, causal_full):
    rng = np.random.default_rng(7 + Hq + L)
    P, D = 16, 32
    K = _rand_bits(rng, (L, Hkv, D))
    V = _rand_bits(rng, (L, Hkv, D))
    q = _rand_bits(rng, (n, Hq, D))
    perm = rng.permutation((L + P - 1) // P + 2)
    kp, vp = _pool_from_contiguous(K, perm, P), _pool_from_contiguous(V, perm, P)
    out = orc.attend(q, kp, vp, perm[None, :].astype(np.int32), np.array([L]),
                     np.array([0, n]), 0.17, Hq, Hkv, P)
    G = Hq // Hkv
    Kf = np.repeat(O.bf16_to_f64(K), G, axis=1)  # query head h <- kv head h // G
    Vf = np.repeat(O.bf16_to_f64(V), G, axis=1)
    qf = O.bf16_to_f64(q)
    if causal_full:   # n == L: bottom-right == top-left causal
        ref = _sdpa(qf, Kf, Vf, 0.17, True)
    else:             # n == 1: decode sees every key
        ref = _sdpa(qf, Kf, Vf, 0.17, False)
    return bool(np.allclose(out, ref, rtol=0, atol=1e-12))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 3), (4, 1)])
def test_decode_matches_sdpa(Hq, Hkv):
    assert check_matches_sdpa(O, Hq, Hkv, L=45, n=1, causal_full=False)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_full_prefill_matches_causal_sdpa(Hq, Hkv):
    assert check_matches_sdpa(O, Hq, Hkv, L=37, n=37, causal_full=True)


# --------------------------------------------------------------------------
# chunked prefill: bottom-right causal alignment
# --------------------------------------------------------------------------

def check_bottom_right_causal(orc):
    rng = np.random.default_rng(8)
    P, D, Hq, Hkv, L, n = 4, 8, 2, 1, 19, 5
    K, V = _rand_bits(rng, (L, Hkv, D)), _rand_bits(rng, (L, Hkv, D))
    q = _rand_bits(rng, (n, Hq, D))
    perm = rng.permutation(8)[:5]
    bt = perm[None, :].astype(np.int32)
    run = lambda K_, V_: orc.attend(q, _pool_from_contiguous(K_, perm, P),
                                    _pool_from_contiguous(V_, perm, P), bt,
                                    np.array([L]), np.array([0, n]), 0.4, Hq, Hkv, P)
    base = run(K, V)
    ok = True
    for j in range(n):
        p = L - n + j
        # a key after position p is invisible to query j ...
        if p + 1 < L:
            K2, V2 = K.copy(), V.copy()
            K2[p + 1] = _rand_bits(rng, (Hkv, D), 5.0)
            V2[p + 1] = _rand_bits(rng, (Hkv, D), 5.0)
            ok &= np.array_equal(run(K2, V2)[j], base[j])
        # ... and the key at position p itself is visible
        V3 = V.copy()
        V3[p] = _rand_bits(rng, (Hkv, D), 5.0)
        ok &= not np.allclose(run(K, V3)[j], base[j])
    # the last query of the chunk is a decode over all L keys
    dec = orc.attend(q[-1:], _pool_from_contiguous(K, perm, P), _pool_from_contiguous(V, perm, P),
                     bt, np.array([L]), np.array([0, 1]), 0.4, Hq, Hkv, P)
    ok &= np.array_equal(dec[0], base[-1])
    return bool(ok)


def test_bottom_right_causal():
    assert check_bottom_right_causal(O)


# --------------------------------------------------------------------------
# brute force: scalar loops with math.exp on a tiny paged batch
# --------------------------------------------------------------------------

def check_brute_force(orc):
    b = make_batch([3, 9, 6], [1, 4, 6], 4, 2, seed=21, pool_factor=1.5)
    P, G = b.page_size, 2
    q = b.q.view(torch.int16).numpy().view(np.uint16)
    kc = b.k_cache.view(torch.int16).numpy().view(np.uint16)
    vc = b.v_cache.view(torch.int16).numpy().view(np.uint16)
    got = orc.attend(q, kc, vc, b.block_tables, b.seq_lens, b.query_start_loc,
                     b.scale, 4, 2, P)
    f = lambda bits: float(np.uint32(int(bits) << 16).view(np.float32))
    worst = 0.0
    for bi in range(b.B):
        L, q0, q1 = int(b.seq_lens[bi]), int(b.query_start_loc[bi]), int(b.query_start_loc[bi + 1])
        n = q1 - q0
        for j in range(n):
            for h in range(4):
                kvh = h // G
                scores = []
                for t in range(L - n + j + 1):
                    page, row = int(b.block_tables[bi][t // P]), t % P
                    scores.append(b.scale * sum(f(q[q0 + j, h, d]) * f(kc[page, kvh, row, d])
                                                for d in range(b.head_dim)))
                mx = max(scores)
                ws = [math.exp(s - mx) for s in scores]
                tot = sum(ws)
                for d in range(0, b.head_dim, 7):
                    acc = 0.0
                    for t, w in enumerate(ws):
                        page, row = int(b.block_tables[bi][t // P]), t % P
                        acc += w * f(vc[page, kvh, row, d])
                    worst = max(worst, abs(acc / tot - got[q0 + j, h, d]))
    return worst < 1e-12


def test_brute_force_loops():
    assert check_brute_force(O)


# --------------------------------------------------------------------------
# split-KV merge algebra
# --------------------------------------------------------------------------

def test_merge_of_any_partition_equals_unsplit():
    rng = np.random.default_rng(9)
    n, D = 300, 32
    q, keys, values = rng.standard_normal(D), rng.standard_normal((n, D)) * 3, rng.standard_normal((n, D))
    ref = O.attend_one(q, keys, values, 0.7)
    for _ in range(20):
        cuts = sorted(set(rng.integers(1, n, size=rng.integers(0, 12)).tolist()))
        parts = O.split_partials(q, keys, values, 0.7, [0] + cuts + [n])
        assert np.allclose(O.merge_partials(parts), ref, rtol=0, atol=1e-12)
    single = O.split_partials(q, keys, values, 0.7, [0, n])
    m, l, o = single[0]
    assert np.allclose(o / l, ref, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# named workloads are well formed (host side only, no tensors)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_workload_structure(idx):
    b = workload(idx, with_tensors=False)
    P = b.page_size
    assert b.query_start_loc[0] == 0 and (np.diff(b.query_start_loc) >= 0).all()
    assert (b.q_lens <= b.seq_lens).all()
    used = set()
    shared = b.info["shared_prefix_pages"]
    for bi in range(b.B):
        pages = b.block_tables[bi, : (int(b.seq_lens[bi]) + P - 1) // P]
        assert ((pages >= 0) & (pages < b.num_blocks)).all()
        own = set(pages[shared:].tolist())
        assert not (own & used), "a page may belong to one sequence only"
        used |= own
    # every new token's slot lies in a page owned by its sequence only
    slot_pages = b.slot_mapping // P
    assert len(set(slot_pages.tolist()) & set(b.block_tables[0, :shared].tolist())) == 0
    expected = {1: (4, 4), 2: (64, 64), 3: (256, 256), 4: (128, 128), 5: (98, 1120)}[idx]
    assert (b.B, b.T) == expected


# --------------------------------------------------------------------------
# planted mistakes: each broken copy of the oracle must fail some pin
# --------------------------------------------------------------------------

def _mutant(**over):
    m = types.ModuleType("mutant")
    m.__dict__.update({k: getattr(O, k) for k in O.__all__})
    m.__dict__.update(over)
    return m


def _attend_variant(kv_map=None, causal=None, scale_mul=1.0, page_map=None):
    def attend(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
               num_q_heads, num_kv_heads, page_size, rows=None):
        G = num_q_heads // num_kv_heads
        T, Hq, D = q.shape
        out = np.full((T, Hq, D), np.nan)
        for b in range(len(seq_lens)):
            q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
            n, L = q1 - q0, int(seq_lens[b])
            if page_map is None:
                K = O.gather(k_cache, block_tables[b], L, page_size)
                V = O.gather(v_cache, block_tables[b], L, page_size)
            else:
                K, V = page_map(k_cache, block_tables[b], L, page_size), page_map(v_cache, block_tables[b], L, page_size)
            for j in range(n):
                p = (L - n + j) if causal is None else causal(L, n, j)
                qr = O.bf16_to_f64(q[q0 + j])
                for h in range(Hq):
                    g = h // G if kv_map is None else kv_map(h, G, num_kv_heads)
                    out[q0 + j, h] = O.attend_one(qr[h], K[: p + 1, g], V[: p + 1, g], scale * scale_mul)
        return out
    return attend


def _swapped_gather(cache, row, L, P):
    j = np.arange(L)
    pages = np.asarray(row)[np.minimum(j % P, len(row) - 1)]
    return O.bf16_to_f64(cache[pages, :, np.minimum(j // P, P - 1), :])


def _all_pins(m):
    return [check_paged_equals_contiguous(m), check_matches_sdpa(m, 8, 2, 45, 1, False),
            check_matches_sdpa(m, 8, 2, 37, 37, True), check_bottom_right_causal(m),
            check_brute_force(m)]


@pytest.mark.parametrize("name,mut", [
    ("kv head h % Hkv", dict(attend=_attend_variant(kv_map=lambda h, G, Hkv: h % Hkv))),
    ("top-left causal", dict(attend=_attend_variant(causal=lambda L, n, j: j))),
    ("scale dropped", dict(attend=_attend_variant(scale_mul=1.0 / 0.17))),
    ("page/row swapped", dict(attend=_attend_variant(page_map=_swapped_gather))),
])
def test_planted_mistakes_are_caught(name, mut):
    assert _all_pins(O) == [True] * 5
    assert not all(_all_pins(_mutant(**mut))), name


def test_planted_write_mistake_is_caught():
    def bad_write(k_new, v_new, slot_mapping, k_cache, v_cache, page_size):
        # page and row swapped: page = s % P, row = s // P
        k_out, v_out = k_cache.copy(), v_cache.copy()
        for t, s in enumerate(slot_mapping):
            if s < 0:
                continue
            page, row = int(s) % page_size, (int(s) // page_size) % page_size
            k_out[page, :, row, :] = k_new[t]
            v_out[page, :, row, :] = v_new[t]
        return k_out, v_out
    assert not check_write_roundtrip(_mutant(write=bad_write))
