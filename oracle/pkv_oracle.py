"""Plain float64 CPU oracle for the paged-KV-cache hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import this module.  The CUDA library never
imports, links or calls it, and it shares no code with the CUDA path: the
only thing both sides consume is the seeded input generator in
``workloads.py``, which holds none of the method's arithmetic.

What the pages fix, and what this oracle follows
------------------------------------------------
* llm-d blog post "What does production-grade LLM inference look like?"
  (introduction): serving engines keep a KV cache and use *paged attention*
  and *continuous batching*; decode is memory-bandwidth-bound and prefill is
  compute-bound.  The post also explains (routing factors; prefix cache
  producers) that a prompt whose prefix is already cached skips that part of
  prefill, i.e. the cached KV pages are reused read-only.
* vLLM notes "EngineCoreClient: dos caminos de cliente, en proceso y
  multiproceso" ("Flujo de datos"): the engine reports ``num_gpu_blocks``
  and the aligned ``block_size`` it reserved, so the cache is a pool of
  fixed-size blocks (pages).
* TensorRT Edge-LLM "HTTP Inference Server Architecture" ("Request
  Lifecycle", "Extension Rules"): the native runtime owns the retained pages
  under a single-writer contract.

The pages print no attention formula, no cache layout and no kernel.  The
readings taken where they are silent:
  * pool layout ``[num_blocks, num_kv_heads, page_size, head_dim]``;
  * ``seq_lens[b]`` counts the tokens written this step;
  * causal alignment is bottom-right: the n queries of sequence b are its last
    n positions ``L-n .. L-1``;
  * grouped-query mapping: query head h reads kv head ``h // (Hq // Hkv)``;
  * ``slot_mapping[t] < 0`` means "no write" (padding);
  * no soft-cap, ALiBi, sliding window or sink tokens.

Attention itself is the textbook definition (scaled dot product, softmax,
weighted sum of values).  Paging and split-KV only reach that same result
faster, so the oracle is that definition written out: gather a sequence's
pages into contiguous K/V, then softmax attention per (query, head).

bf16 data are handled as their raw ``uint16`` bit patterns; a bf16 value is by
definition the binary32 whose upper 16 bits are those bits.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64",
    "write",
    "export_pages",
    "import_pages",
    "gather",
    "attend",
    "attend_one",
    "split_partials",
    "merge_partials",
    "e4m3_to_f64",
    "e4m3_encode",
    "row_scale_exponent",
    "quantize_rows",
    "write_fp8",
    "gather_fp8",
    "attend_fp8",
]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64.

    bf16 is the top half of an IEEE-754 binary32, so shifting the 16 bits into
    the high half of a uint32 and reinterpreting gives the value exactly.
    """
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns")
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def write(k_new, v_new, slot_mapping, k_cache, v_cache, page_size):
    """Step a1 -- scatter new K/V rows into the page pool through slot_mapping.

    Token t with slot s >= 0 lands in page ``s // page_size``, row
    ``s % page_size`` of every kv head; s < 0 is skipped.  Tokens are applied in
    ascending t.  Returns new (k_cache, v_cache) arrays; the inputs are not
    modified.  Pure copy of bit patterns, so the result is exact.

    Shapes: k_new/v_new [T, Hkv, D] uint16; slot_mapping [T] int64;
    k_cache/v_cache [NB, Hkv, P, D] uint16.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    num_blocks = k_out.shape[0]
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        page, row = divmod(int(s), int(page_size))
        if page >= num_blocks:
            raise IndexError(f"slot {int(s)} of token {t} is outside the pool")
        k_out[page, :, row, :] = k_new[t]
        v_out[page, :, row, :] = v_new[t]
    return k_out, v_out


def export_pages(k_cache, v_cache, pages):
    """Whole pages in transfer order: [n, 2 (K, V), Hkv, P, D] bit patterns.

    A disaggregated prefill engine hands a request's KV pages to the decode
    engine (llm-d blog, P/D disaggregation); this is the content moved.
    """
    pages = np.asarray(pages, dtype=np.int64)
    return np.stack([np.asarray(k_cache)[pages], np.asarray(v_cache)[pages]], axis=1)


def import_pages(buf, pages, k_cache, v_cache):
    """Inverse of export_pages: returns new (k_cache, v_cache) with the
    listed pages replaced by the buffer's content (later duplicates win)."""
    k_out, v_out = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    for i, pg in enumerate(np.asarray(pages, dtype=np.int64)):
        k_out[pg] = buf[i, 0]
        v_out[pg] = buf[i, 1]
    return k_out, v_out


def gather(cache, block_table_row, seq_len, page_size):
    """Step a2 -- contiguous float64 copy of one sequence's cached rows.

    Logical token j of the sequence is stored in page
    ``block_table_row[j // page_size]`` at row ``j % page_size``.
    Returns [seq_len, Hkv, D] float64.
    """
    j = np.arange(int(seq_len))
    pages = np.asarray(block_table_row)[j // page_size]
    rows = j % page_size
    # cache[pages, :, rows, :] pairs pages[i] with rows[i] -> shape [L, Hkv, D]
    return bf16_to_f64(cache[pages, :, rows, :])


def attend_one(q_vec, keys, values, scale):
    """Softmax attention of one query vector over visible keys (float64).

    s_t = scale * <q, k_t>;  w = exp(s - max s) / sum exp(s - max s);
    out = sum_t w_t v_t.
    Shapes: q_vec [D], keys/values [n_visible, D].
    """
    s = scale * (keys @ q_vec)
    w = np.exp(s - s.max())
    w = w / w.sum()
    return w @ values


def attend(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
           num_q_heads, num_kv_heads, page_size, rows=None):
    """Steps a2-a5 -- paged attention of a continuous batch, float64 result.

    Sequence b owns query rows ``query_start_loc[b] .. query_start_loc[b+1]-1``
    (n of them) and has L = seq_lens[b] cached tokens, the new ones included.
    Query j of the sequence sits at position p = L - n + j and sees keys
    0..p (bottom-right causal; with n = 1 this is plain decode over all L
    keys).  Query head h uses kv head h // (num_q_heads // num_kv_heads).

    ``q`` is [T, Hq, D] uint16 (bf16 bits); caches [NB, Hkv, P, D] uint16.
    ``scale`` is widened to float64 as given.  If ``rows`` is given, only those
    query rows are computed (others stay NaN) -- used to sample big batches.
    Returns [T, Hq, D] float64.
    """
    def fetch(b, L):
        return (gather(k_cache, block_tables[b], L, page_size),
                gather(v_cache, block_tables[b], L, page_size))
    return _attend_batch(q, fetch, seq_lens, query_start_loc, scale, num_q_heads,
                         num_kv_heads, rows)


def _attend_batch(q, fetch, seq_lens, query_start_loc, scale, num_q_heads,
                  num_kv_heads, rows):
    """The per-sequence loop of attend; fetch(b, L) returns sequence b's
    gathered float64 K and V, each [L, Hkv, D]."""
    if num_q_heads % num_kv_heads != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = num_q_heads // num_kv_heads
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    T, Hq, D = q.shape
    out = np.full((T, Hq, D), np.nan, dtype=np.float64)
    want = None if rows is None else set(int(r) for r in rows)
    scale = float(np.float64(scale))
    for b in range(len(lens)):
        q0, q1 = int(qsl[b]), int(qsl[b + 1])
        n, L = q1 - q0, int(lens[b])
        if n == 0:
            continue
        if n > L:
            raise ValueError(f"sequence {b}: {n} queries but only {L} tokens")
        if want is not None and not any(r in want for r in range(q0, q1)):
            continue
        K, V = fetch(b, L)
        for j in range(n):
            if want is not None and (q0 + j) not in want:
                continue
            p = L - n + j
            qrow = bf16_to_f64(q[q0 + j])
            for h in range(Hq):
                g = h // group
                out[q0 + j, h] = attend_one(qrow[h], K[: p + 1, g], V[: p + 1, g], scale)
    return out


def split_partials(q_vec, keys, values, scale, bounds):
    """Split-KV partial states of one (query, head) over key ranges.

    ``bounds`` = [b0=0, b1, ..., bk=n_visible].  For each range [b_i, b_i+1)
    returns (m_i, l_i, o_i): the range's score maximum, the sum of
    exp(s - m_i), and the unnormalised sum of exp(s - m_i) * v.
    """
    s = scale * (keys @ q_vec)
    parts = []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        if hi <= lo:
            continue
        m = s[lo:hi].max()
        e = np.exp(s[lo:hi] - m)
        parts.append((m, e.sum(), e @ values[lo:hi]))
    return parts


def merge_partials(parts):
    """Step a4 -- log-sum-exp merge of split partial states.

    M = max_i m_i;  out = sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i.
    """
    M = max(m for m, _, _ in parts)
    num = sum(np.exp(m - M) * o for m, _, o in parts)
    den = sum(np.exp(m - M) * l for m, l, _ in parts)
    return num / den


# ---------------------------------------------------------------------------
# FP8 (e4m3) pages
# ---------------------------------------------------------------------------
# The pages do not describe 8-bit KV pages; this part follows the OCP "8-bit
# Floating Point Specification (OFP8)", format E4M3: 1 sign bit, 4 exponent
# bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
# m * 2^-9; S.1111.111 is NaN; there are no infinities, so the largest finite
# magnitude is 1.75 * 2^8 = 448.
#
# Readings taken here:
#   * one scale per (page, kv head, row): a page fills one token per decode
#     step, so a single per-page scale would force re-encoding rows already
#     stored whenever a later token raised the page's maximum; a per-row scale
#     keeps the write a pure scatter.  The 16 scales of a (page, kv head) are
#     stored next to its codes.
#   * the scale is a power of two 2^e, stored as the byte e + 127 (as in the
#     E8M0 scale type of the OCP microscaling formats), with e the smallest
#     integer for which max|x| <= 448 * 2^e, clamped to [-126, 127];
#     x * 2^-e is then exact and the only rounding is the E4M3 one.
#   * rounding is to nearest, ties to the even code; the sign is kept, so a
#     negative value that rounds to zero gives the code 0x80 (-0).

E4M3_MAX = 448.0


def e4m3_to_f64(codes):
    """Exact value of E4M3 codes (uint8 array) as float64; 0x7F/0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    expo = (c >> 3) & 0xF
    mant = c & 0x7
    mag = np.where(expo == 0, mant * 2.0 ** -9, (1.0 + mant / 8.0) * np.exp2(expo - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where((c & 0x80) != 0, -mag, mag)


_E4M3_POS = None


def _e4m3_positive_table():
    """Values of codes 0x00..0x7E (non-negative, finite), increasing."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    return _E4M3_POS


def e4m3_encode(x):
    """Nearest E4M3 code of float64 values with |x| <= 448 (ties to the even
    code, sign kept).  Raises for non-finite or out-of-range input."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)) or np.any(np.abs(x) > E4M3_MAX):
        raise ValueError("e4m3_encode takes finite values with |x| <= 448")
    table = _e4m3_positive_table()
    a = np.abs(x)
    lo = np.searchsorted(table, a, side="right") - 1      # largest code value <= a
    hi = np.minimum(lo + 1, 0x7E)
    d_lo, d_hi = a - table[lo], table[hi] - a
    take_hi = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)))
    code = np.where(take_hi, hi, lo).astype(np.int64)
    code = code | (np.signbit(x).astype(np.int64) << 7)
    return code.astype(np.uint8)


def row_scale_exponent(amax):
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-126, 127]."""
    amax = float(amax)
    if amax == 0.0:
        return -126
    e = int(np.floor(np.log2(amax / E4M3_MAX)))
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    while amax <= E4M3_MAX * 2.0 ** (e - 1):
        e -= 1
    return min(max(e, -126), 127)


def quantize_rows(x_bits):
    """E4M3 codes and scale bytes of bf16 rows.

    ``x_bits`` [..., D] uint16 (bf16 bits).  Each row (last axis) gets
    e = row_scale_exponent(max |x|); its codes are e4m3_encode(x * 2^-e) and
    its scale byte is e + 127.  Returns (codes [..., D] uint8, scale [...] uint8).
    """
    x = bf16_to_f64(x_bits)
    amax = np.abs(x).max(axis=-1)
    e = np.vectorize(row_scale_exponent, otypes=[np.int64])(amax)
    codes = e4m3_encode(x * np.exp2(-e.astype(np.float64))[..., None])
    return codes, (e + 127).astype(np.uint8)


def write_fp8(k_new, v_new, slot_mapping, k_codes, v_codes, k_scale, v_scale, page_size):
    """KV write into FP8 pages: each new (token, kv head) row of K and of V is
    quantised with quantize_rows and scattered like ``write``; its scale byte
    goes to [page, head, row] of k_scale / v_scale.

    Shapes: k_new/v_new [T, Hkv, D] uint16; codes [NB, Hkv, P, D] uint8;
    scales [NB, Hkv, P] uint8.  Returns new (k_codes, v_codes, k_scale, v_scale).
    """
    kc, vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    ks, vs = np.array(k_scale, copy=True), np.array(v_scale, copy=True)
    kq, kqs = quantize_rows(np.asarray(k_new))
    vq, vqs = quantize_rows(np.asarray(v_new))
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        page, row = divmod(int(s), int(page_size))
        if page >= kc.shape[0]:
            raise IndexError(f"slot {int(s)} of token {t} is outside the pool")
        kc[page, :, row, :], ks[page, :, row] = kq[t], kqs[t]
        vc[page, :, row, :], vs[page, :, row] = vq[t], vqs[t]
    return kc, vc, ks, vs


def gather_fp8(codes, scales, block_table_row, seq_len, page_size):
    """Contiguous float64 values of one sequence's FP8 rows: code value times
    2^(scale byte - 127).  Returns [seq_len, Hkv, D]."""
    j = np.arange(int(seq_len))
    pages = np.asarray(block_table_row)[j // page_size]
    rows = j % page_size
    val = e4m3_to_f64(codes[pages, :, rows, :])
    return val * np.exp2(scales[pages, :, rows].astype(np.float64) - 127.0)[..., None]


def attend_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, seq_lens,
               query_start_loc, scale, num_q_heads, num_kv_heads, page_size, rows=None):
    """attend() over FP8 pages: the same textbook attention, with K and V the
    exact values the codes and scales stand for."""
    def fetch(b, L):
        return (gather_fp8(k_codes, k_scale, block_tables[b], L, page_size),
                gather_fp8(v_codes, v_scale, block_tables[b], L, page_size))
    return _attend_batch(q, fetch, seq_lens, query_start_loc, scale, num_q_heads,
                         num_kv_heads, rows)
