"""Pins of the oracle's FP8 (E4M3) page functions, each against something other
than the oracle itself: the format's closed-form values (OCP 8-bit Floating
Point Specification, E4M3), PyTorch's independent float8_e4m3fn conversion,
the rounding error bound of a 3-bit mantissa, and torch SDPA on contiguous
dequantised K/V.  Broken copies of the functions (planted mistakes) must fail
some pin.  CPU only.
"""

import numpy as np
import pytest
import torch

import oracle.pkv_oracle as O


def _all_bf16_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        x = O.bf16_to_f64(bits)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    return bits[keep], x[keep]


def _torch_e4m3(x_f64):
    return torch.from_numpy(np.asarray(x_f64, dtype=np.float64)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _rand_rows(rng, shape, spread=6.0):
    """bf16 rows whose magnitudes span many binades (per-row and per-element)."""
    row_scale = np.exp2(rng.uniform(-spread, spread, size=shape[:-1] + (1,)))
    x = rng.standard_normal(shape) * row_scale * np.exp2(rng.uniform(-3, 3, size=shape))
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- the format

def check_e4m3_values(orc):
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x7D: 416.0,
             0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    v = orc.e4m3_to_f64(np.array(list(known), dtype=np.uint8))
    if not np.array_equal(v, np.array(list(known.values()))):
        return False
    neg0 = orc.e4m3_to_f64(np.array([0x80], dtype=np.uint8))[0]
    nans = orc.e4m3_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))
    return neg0 == 0.0 and np.signbit(neg0) and np.all(np.isnan(nans))


def test_e4m3_closed_form_values():
    assert check_e4m3_values(O)


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.e4m3_to_f64(codes), ref)
    assert np.array_equal(np.signbit(O.e4m3_to_f64(codes)), np.signbit(ref))


def check_encode_matches_torch(orc):
    b, x = _all_bf16_in_range()
    return bool(np.array_equal(orc.e4m3_encode(x), _torch_e4m3(x)))


def test_e4m3_encode_matches_torch_on_every_bf16_value():
    """Every finite bf16 value with |x| <= 448 (34,754 of them)."""
    assert check_encode_matches_torch(O)


def check_ties(orc):
    cases = {1.0625: 0x38,           # halfway 1.0 | 1.125 -> even mantissa 000
             1.1875: 0x3A,           # halfway 1.125 | 1.25 -> 010
             2.0 ** -10: 0x00,       # halfway 0 | 2^-9 -> 0
             3 * 2.0 ** -10: 0x02,   # halfway 2^-9 | 2^-8 -> code 2
             432.0: 0x7E,            # halfway 416 | 448 -> 448 (110)
             -1.0625: 0xB8,
             -(2.0 ** -11): 0x80,    # rounds to zero, sign kept
             1.05: 0x38, 1.07: 0x39, 1.1325: 0x39}
    got = orc.e4m3_encode(np.array(list(cases)))
    return bool(np.array_equal(got, np.array(list(cases.values()), dtype=np.uint8)))


def test_e4m3_ties_to_even_and_signed_zero():
    assert check_ties(O)


def test_e4m3_encode_rejects_out_of_range():
    with pytest.raises(ValueError):
        O.e4m3_encode(np.array([448.5]))
    with pytest.raises(ValueError):
        O.e4m3_encode(np.array([np.nan]))


# ---------------------------------------------------------------- the scale

def check_scale_exponent(orc):
    cases = {448.0: 0, 450.0: 1, 1.0: -8, 1.75: -8, 1.7578125: -7, 224.0: -1, 896.0: 1,
             0.0: -126, 2.0 ** -133: -126, 3.0e38: 120}
    return all(orc.row_scale_exponent(a) == e for a, e in cases.items())


def test_scale_exponent_closed_forms():
    assert check_scale_exponent(O)


def test_scaled_row_maximum_lands_in_the_top_binade():
    """For every unclamped row, max|x| / 2^e lies in (224, 448]."""
    rng = np.random.default_rng(7)
    x = O.bf16_to_f64(_rand_rows(rng, (400, 128), spread=40.0))
    for row in x:
        a = np.abs(row).max()
        e = O.row_scale_exponent(a)
        assert 224.0 < a / 2.0 ** e <= 448.0


def check_roundtrip_bound(orc):
    """Round to nearest of a 3-bit mantissa: error <= 2^-4 |x| for scaled values
    in the normal range (>= 2^-6), <= 2^-10 (scaled units) below it."""
    rng = np.random.default_rng(3)
    xb = _rand_rows(rng, (64, 3, 128))
    codes, sc = orc.quantize_rows(xb)
    x = O.bf16_to_f64(xb)
    unit = np.exp2(sc.astype(np.float64) - 127.0)[..., None]
    deq = O.e4m3_to_f64(codes) * unit
    err = np.abs(deq - x)
    scaled = np.abs(x) / unit
    bound = np.where(scaled >= 2.0 ** -6, 2.0 ** -4 * np.abs(x), 2.0 ** -10 * unit)
    # the largest code of every row sits in the top binade [224, 448]
    top = (np.abs(deq) / unit).max(axis=-1)
    return bool(np.all(err <= bound) and np.all(top >= 224.0) and codes.dtype == np.uint8)


def test_quantize_roundtrip_error_bound():
    assert check_roundtrip_bound(O)


def test_quantize_zero_and_negative_zero_rows():
    z = np.zeros((2, 128), dtype=np.uint16)
    z[1, :] = 0x8000  # -0.0
    codes, sc = O.quantize_rows(z)
    assert np.all(sc == 1) and np.all(codes[0] == 0) and np.all(codes[1] == 0x80)


# ---------------------------------------------------------------- write

def check_write_fp8(orc):
    rng = np.random.default_rng(11)
    NB, Hkv, P, D, T = 6, 2, 16, 128, 9
    kc = rng.integers(0, 256, size=(NB, Hkv, P, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, P, D), dtype=np.uint8)
    ks = rng.integers(0, 256, size=(NB, Hkv, P), dtype=np.uint8)
    vs = rng.integers(0, 256, size=(NB, Hkv, P), dtype=np.uint8)
    kn, vn = _rand_rows(rng, (T, Hkv, D)), _rand_rows(rng, (T, Hkv, D))
    slots = np.array([5, -1, 17, 95, 0, -3, 40, 41, 63], dtype=np.int64)
    k2, v2, ks2, vs2 = orc.write_fp8(kn, vn, slots, kc, vc, ks, vs, P)
    touched = np.zeros((NB, P), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        pg, r = divmod(int(s), P)
        touched[pg, r] = True
        for cache, sc, new in ((k2, ks2, kn), (v2, vs2, vn)):
            x = O.bf16_to_f64(new[t])
            unit = np.exp2(sc[pg, :, r].astype(np.float64) - 127.0)[:, None]
            deq = O.e4m3_to_f64(cache[pg, :, r, :]) * unit
            if not np.all(np.abs(deq - x) <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * unit)):
                return False
    keep = ~touched
    return bool(np.array_equal(k2.transpose(0, 2, 1, 3)[keep], kc.transpose(0, 2, 1, 3)[keep])
                and np.array_equal(vs2.transpose(0, 2, 1)[keep], vs.transpose(0, 2, 1)[keep])
                and np.array_equal(ks2.transpose(0, 2, 1)[keep], ks.transpose(0, 2, 1)[keep]))


def test_write_fp8_places_rows_and_leaves_the_rest():
    assert check_write_fp8(O)


# ---------------------------------------------------------------- attention

def check_attend_fp8_matches_sdpa(orc):
    """Paged FP8 attention equals SDPA (float64) on contiguous K/V decoded by
    torch's own float8 conversion, under a shuffled block table."""
    rng = np.random.default_rng(5)
    Hq, Hkv, D, P, L = 8, 2, 128, 16, 53
    npg = (L + P - 1) // P
    kb, vb = _rand_rows(rng, (L, Hkv, D), 2.0), _rand_rows(rng, (L, Hkv, D), 2.0)
    kq, ksc = O.quantize_rows(kb)
    vq, vsc = O.quantize_rows(vb)
    perm = rng.permutation(npg + 3)[:npg]
    NB = npg + 3
    kc = np.full((NB, Hkv, P, D), 0x7F, dtype=np.uint8)   # NaN canaries
    vc = np.full((NB, Hkv, P, D), 0x7F, dtype=np.uint8)
    ks = np.full((NB, Hkv, P), 200, dtype=np.uint8)
    vs = np.full((NB, Hkv, P), 200, dtype=np.uint8)
    for j in range(L):
        kc[perm[j // P], :, j % P], ks[perm[j // P], :, j % P] = kq[j], ksc[j]
        vc[perm[j // P], :, j % P], vs[perm[j // P], :, j % P] = vq[j], vsc[j]
    q = _rand_rows(rng, (1, Hq, D), 0.5)
    scale = 1 / np.sqrt(D)
    out = orc.attend_fp8(q, kc, vc, ks, vs, perm[None, :], np.array([L]), np.array([0, 1]),
                         scale, Hq, Hkv, P)

    def deq(codes, sc):
        v = torch.from_numpy(codes).view(torch.float8_e4m3fn).double()
        return v * torch.from_numpy(np.exp2(sc.astype(np.float64) - 127.0))[..., None]
    K, V = deq(kq, ksc), deq(vq, vsc)                       # [L, Hkv, D]
    Q = torch.from_numpy(O.bf16_to_f64(q[0]))               # [Hq, D]
    Kx = K.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    Vx = V.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q[:, None, :], Kx, Vx, scale=scale)[:, 0]
    return bool(np.allclose(out[0], ref.numpy(), rtol=0, atol=1e-12))


def test_attend_fp8_matches_sdpa_on_dequantised_values():
    assert check_attend_fp8_matches_sdpa(O)


# ---------------------------------------------------------------- planted mistakes

def _mutant(**over):
    import types
    m = types.ModuleType("mutant_fp8")
    m.__dict__.update({k: getattr(O, k) for k in O.__all__})
    m.__dict__.update(over)
    return m


def _encode_truncating(x):
    x = np.asarray(x, dtype=np.float64)
    t = O._e4m3_positive_table()
    code = np.searchsorted(t, np.abs(x), side="right") - 1
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    t = O._e4m3_positive_table()
    a = np.abs(x)
    lo = np.searchsorted(t, a, side="right") - 1
    hi = np.minimum(lo + 1, 0x7E)
    code = np.where((hi != lo) & (t[hi] - a <= a - t[lo]), hi, lo)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def _scale_one_low(amax):
    return O.row_scale_exponent(amax) - 1 if amax > 0 else -126


def _gather_ignoring_scale(codes, scales, row, L, P):
    j = np.arange(int(L))
    return O.e4m3_to_f64(codes[np.asarray(row)[j // P], :, j % P, :])


def _e4m3_bias_8(codes):
    return O.e4m3_to_f64(codes) / 2.0


def _pins(m):
    return [check_e4m3_values(m), check_encode_matches_torch(m), check_ties(m),
            check_scale_exponent(m), check_write_fp8(m), check_attend_fp8_matches_sdpa(m)]


def _quantize_with(scale_fn, encode_fn):
    def quantize_rows(x_bits):
        x = O.bf16_to_f64(x_bits)
        e = np.vectorize(scale_fn, otypes=[np.int64])(np.abs(x).max(axis=-1))
        xs = np.clip(x * np.exp2(-e.astype(np.float64))[..., None], -448, 448)
        return encode_fn(xs), (e + 127).astype(np.uint8)
    return quantize_rows


@pytest.mark.parametrize("name,mut", [
    ("truncating rounding", dict(e4m3_encode=_encode_truncating)),
    ("ties away from zero", dict(e4m3_encode=_encode_ties_away)),
    ("scale exponent one too low", dict(row_scale_exponent=_scale_one_low,
                                        quantize_rows=_quantize_with(_scale_one_low, O.e4m3_encode))),
    ("scale ignored when reading", dict(gather_fp8=_gather_ignoring_scale,
                                        attend_fp8=None)),
    ("exponent bias 8", dict(e4m3_to_f64=_e4m3_bias_8)),
])
def test_planted_fp8_mistakes_are_caught(name, mut):
    assert _pins(O) == [True] * 6
    if "attend_fp8" in mut:
        # rebuild attend_fp8 on top of the broken gather
        g = mut["gather_fp8"]

        def attend_fp8(q, kc, vc, ks, vs, bt, lens, qsl, scale, Hq, Hkv, P, rows=None):
            def fetch(b, L):
                return g(kc, ks, bt[b], L, P), g(vc, vs, bt[b], L, P)
            return O._attend_batch(q, fetch, lens, qsl, scale, Hq, Hkv, rows)
        mut = dict(mut, attend_fp8=attend_fp8)
    assert not all(_pins(_mutant(**mut))), name
