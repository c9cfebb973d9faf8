"""FP8 (E4M3) pages: pkv_write_fp8 bit-exact against the oracle's write_fp8
(codes and scale bytes, whole pools), pkv_attend_fp8 within the attention
tolerance of the oracle's attend_fp8 (the exact values the codes stand for).
"""

import numpy as np
import pytest
import torch

import oracle.pkv_oracle as O
import paged_kv_cache_pkv_gb300 as pkv
from helpers import bits, compare, compare_large_outputs, to_device
from workloads import fp8_pools, large_value_rows, make_batch, workload

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.detach().contiguous().cpu().numpy()


def _gpu_write(batch, pools, meta=None, k_new=None, v_new=None):
    meta = meta or to_device(batch)
    kc, vc, ks, vs = (p.clone() for p in pools)
    pkv.write_fp8(batch.k_new if k_new is None else k_new, batch.v_new if v_new is None else v_new,
                  meta["slot_mapping"], kc, vc, ks, vs)
    torch.cuda.synchronize()
    return kc, vc, ks, vs


def _oracle_write(batch, pools, k_new=None, v_new=None):
    kn = bits(batch.k_new if k_new is None else k_new)
    vn = bits(batch.v_new if v_new is None else v_new)
    return O.write_fp8(kn, vn, batch.slot_mapping, *(_u8(p) for p in pools), batch.page_size)


def _run(batch, seed, rows=None, what="", v_values=None, cmp=compare):
    pools = fp8_pools(batch, seed, v_values=v_values)
    meta = to_device(batch)
    kc, vc, ks, vs = _gpu_write(batch, pools, meta)
    out = pkv.attend_fp8(batch.q, kc, vc, ks, vs, meta["block_tables"], meta["seq_lens"],
                         meta["query_start_loc"], batch.scale)
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    ref = _oracle_write(batch, pools)
    for got, want in zip((kc, vc, ks, vs), ref):
        assert np.array_equal(_u8(got), want)
    expected = O.attend_fp8(bits(batch.q), *ref, batch.block_tables, batch.seq_lens,
                            batch.query_start_loc, batch.scale, batch.num_q_heads,
                            batch.num_kv_heads, batch.page_size, rows=rows)
    return cmp(out, expected, rows=rows, what=what or batch.name)


# ---------------------------------------------------------------- write

@pytest.mark.parametrize("idx", [1, 2, 5])
def test_write_fp8_bit_exact_named(pkvlib, idx):
    b = workload(idx, device="cuda")
    pools = fp8_pools(b, 77 + idx)
    got = _gpu_write(b, pools)
    for g, w, name in zip(got, _oracle_write(b, pools), ("k codes", "v codes", "k scale", "v scale")):
        assert np.array_equal(_u8(g), w), name
    assert pkv.get_last_error() == 0


def test_write_fp8_special_rows(pkvlib):
    """Rows that exercise every branch of the encoding: zeros, -0, bf16
    subnormals, the largest bf16, exact ties of the E4M3 grid, maxima just
    above and at 448 * 2^k, single-spike rows, and ordinary rows."""
    rng = np.random.default_rng(21)
    T, Hkv, D = 24, 2, 128
    x = (rng.standard_normal((T, Hkv, D)) * np.exp2(rng.uniform(-20, 20, (T, Hkv, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2, 0] = np.float32(2.0 ** -133) * np.arange(1, D + 1, dtype=np.float32)  # bf16 subnormals
    x[3, 0] = 3.3e38
    x[3, 1] = -3.3e38 * np.linspace(0, 1, D)
    grid = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 432.0, 1.0, 448.0, -1.0625])
    x[4, 0] = np.resize(grid, D) * 2.0 ** 5  # row max 448 * 2^5: e = 5, ties survive scaling
    x[4, 1] = np.resize(grid, D) * 2.0 ** -20
    x[5, 0] = 0.0
    x[5, 0, 17] = 450.0  # max just above 448 -> e = 1
    x[5, 1] = 0.0
    x[5, 1, 3] = -448.0
    x[6] = -np.abs(x[6]) * 1e-3  # negative values, some rounding to -0
    t = torch.from_numpy(x).to(torch.bfloat16)
    b = make_batch([16] * 3 + [40] * 3, [1, 1, 1, 1, 1, 19], 4, Hkv, seed=22, device="cuda")
    assert b.T == T
    k_new = t.cuda()
    v_new = (-t).cuda()
    pools = fp8_pools(b, 23)
    got = _gpu_write(b, pools, k_new=k_new, v_new=v_new)
    for g, w, name in zip(got, _oracle_write(b, pools, k_new=k_new, v_new=v_new),
                          ("k codes", "v codes", "k scale", "v scale")):
        assert np.array_equal(_u8(g), w), name


def test_write_fp8_padding_and_bad_slot(pkvlib):
    b = make_batch([5, 33, 16, 40], [2, 1, 16, 3], 4, 2, seed=24, device="cuda")
    slots = b.slot_mapping.copy()
    slots[[0, 5]] = -1
    slots[7] = b.num_blocks * 16 + 3  # outside the pool: skipped and flagged
    meta = to_device(b)
    meta["slot_mapping"] = torch.from_numpy(slots).cuda()
    pools = fp8_pools(b, 25)
    got = _gpu_write(b, pools, meta)
    assert pkv.get_last_error() & pkv.STATUS_BAD_SLOT
    good = slots.copy()
    good[7] = -1
    ref = O.write_fp8(bits(b.k_new), bits(b.v_new), good, *(_u8(p) for p in pools), 16)
    for g, w in zip(got, ref):
        assert np.array_equal(_u8(g), w)


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("idx", [1, 2])
def test_attend_fp8_named_all_rows(pkvlib, idx):
    _run(workload(idx, device="cuda"), 90 + idx)


def test_attend_fp8_long_tail_rows(pkvlib):
    from test_attend import long_tail_rows
    b = workload(3, device="cuda")
    _run(b, 93, rows=long_tail_rows(b, seed=3), what="cfg3 fp8 64 rows")


def test_attend_fp8_mixed_step_all_rows(pkvlib):
    """Every row: prefill chunks of 512 rows on the tensor-core kernel,
    decode rows on split-KV, FP8 pages."""
    b = workload(5, device="cuda")
    _run(b, 95, what="cfg5 fp8 all rows")


@pytest.mark.parametrize("seed", range(4))
def test_attend_fp8_random_small_batches(pkvlib, seed):
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 9))
    lens = rng.integers(1, 301, size=B)
    qlens = np.array([int(rng.integers(1, min(40, L) + 1)) if rng.random() < 0.4 else 1 for L in lens])
    hq, hkv = [(8, 2), (32, 8), (4, 4), (16, 2)][seed]
    _run(make_batch(lens, qlens, hq, hkv, seed=seed + 50, device="cuda"), seed)


def test_attend_fp8_stale_rows_do_not_leak(pkvlib):
    """Rows past a sequence's length hold NaN codes and scale bytes 0 and 255;
    none of them may reach the output."""
    b = make_batch([17, 33, 250, 64], [1, 4, 1, 20], 8, 2, seed=31, device="cuda")
    kc, vc, ks, vs = fp8_pools(b, 32)
    for bi in range(b.B):
        L = int(b.seq_lens[bi])
        last = int(b.block_tables[bi, (L - 1) // 16])
        if L % 16:
            kc[last, :, L % 16:, :] = 0x7F
            vc[last, :, L % 16:, :] = 0xFF
            ks[last, :, L % 16:] = 255
            vs[last, :, L % 16:] = 0
    pools = (kc, vc, ks, vs)
    meta = to_device(b)
    g = _gpu_write(b, pools, meta)
    out = pkv.attend_fp8(b.q, *g, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale)
    torch.cuda.synchronize()
    ref = _oracle_write(b, pools)
    expected = O.attend_fp8(bits(b.q), *ref, b.block_tables, b.seq_lens, b.query_start_loc, b.scale,
                            b.num_q_heads, b.num_kv_heads, b.page_size)
    compare(out, expected, what="fp8 stale")


@pytest.mark.parametrize("hq,hkv,L,n", [(32, 8, 1100, 130), (16, 2, 257, 257), (8, 8, 640, 300),
                                        (32, 2, 129, 33), (64, 4, 3000, 17), (32, 8, 2000, 100),
                                        (16, 8, 700, 200)])
def test_attend_fp8_prefill_chunks_all_rows(pkvlib, hq, hkv, L, n):
    """Chunks longer than the split-KV bound run on the tensor-core kernel, the
    pages widened exactly to bf16 in shared memory; every row."""
    b = make_batch([L, 40], [n, 1], hq, hkv, seed=L + n + 7, device="cuda")
    tr = pkv.Trace(64)
    with tr:
        _run(b, L + n, what=f"fp8 prefill {hq}/{hkv} L={L} n={n}")
    counts = {k: tr.read(k)[1] for k in ("decode", "prefill")}
    tr.close()
    assert counts["prefill"] == 1


@pytest.mark.parametrize("lens,qlens", [
    ([2048, 64], [512, 1]),                   # long prefill chunk, short split-KV work
    ([3000] * 40 + [300], [1] * 40 + [200]),  # long split-KV work, short prefill chunk
])
def test_attend_fp8_mixed_step_result_is_stream_ordered(pkvlib, lens, qlens):
    """A copy ordered on the stream right after pkv_attend_fp8 (no device-wide
    synchronisation) reads the complete output, whichever kernel ends last."""
    b = make_batch(lens, qlens, 32, 8, seed=sum(lens) + 1, device="cuda")
    pools = fp8_pools(b, 41)
    meta = to_device(b)
    g = _gpu_write(b, pools, meta)
    out = torch.full_like(b.q, float("nan"))
    torch.cuda.synchronize()
    pkv.attend_fp8(b.q, *g, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
                   out=out)
    host = out.cpu()  # stream-ordered copy
    assert pkv.get_last_error() == 0
    ref = _oracle_write(b, pools)
    expected = O.attend_fp8(bits(b.q), *ref, b.block_tables, b.seq_lens, b.query_start_loc, b.scale,
                            b.num_q_heads, b.num_kv_heads, b.page_size)
    compare(host, expected, what=f"fp8 stream-ordered read {len(lens)} rows")


def test_attend_fp8_prefill_stale_rows_do_not_leak(pkvlib):
    """A prefill chunk whose last page is partly past the sequence: those rows
    hold NaN codes and scale bytes 0 and 255, and must not reach the output."""
    b = make_batch([17, 150, 250], [1, 40, 1], 8, 2, seed=33, device="cuda")
    kc, vc, ks, vs = fp8_pools(b, 34)
    for bi in range(b.B):
        L = int(b.seq_lens[bi])
        last = int(b.block_tables[bi, (L - 1) // 16])
        if L % 16:
            kc[last, :, L % 16:, :] = 0x7F
            vc[last, :, L % 16:, :] = 0xFF
            ks[last, :, L % 16:] = 255
            vs[last, :, L % 16:] = 0
    pools = (kc, vc, ks, vs)
    meta = to_device(b)
    g = _gpu_write(b, pools, meta)
    out = pkv.attend_fp8(b.q, *g, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale)
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    ref = _oracle_write(b, pools)
    expected = O.attend_fp8(bits(b.q), *ref, b.block_tables, b.seq_lens, b.query_start_loc, b.scale,
                            b.num_q_heads, b.num_kv_heads, b.page_size)
    compare(out, expected, what="fp8 prefill stale")


def _cascade_fp8(batch, prefix_pages, seed, max_query_len=0, rows=None):
    pools = fp8_pools(batch, seed)
    meta = to_device(batch)
    kc, vc, ks, vs = _gpu_write(batch, pools, meta)
    out = pkv.attend_fp8(batch.q, kc, vc, ks, vs, meta["block_tables"], meta["seq_lens"],
                         meta["query_start_loc"], batch.scale, max_query_len=max_query_len,
                         shared_prefix_pages=prefix_pages)
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    ref = _oracle_write(batch, pools)
    expected = O.attend_fp8(bits(batch.q), *ref, batch.block_tables, batch.seq_lens,
                            batch.query_start_loc, batch.scale, batch.num_q_heads,
                            batch.num_kv_heads, batch.page_size, rows=rows)
    return out, expected


def test_attend_fp8_cascade_prefix_shared_workload(pkvlib):
    """Config 4 on FP8 pages: 128 sequences on one 2048-token prefix, the
    prefix attended once per kv head by the tensor-core prefix pass."""
    b = workload(4, device="cuda")
    out, expected = _cascade_fp8(b, b.info["shared_prefix_pages"], 97, max_query_len=1)
    compare(out, expected, what="fp8 cascade cfg4 all rows")


@pytest.mark.parametrize("hq,hkv,prefix,suffixes", [
    (32, 8, 80, [1, 17, 100, 16]),
    (16, 2, 1600, [3, 250, 33]),
    (64, 8, 512, [70, 5]),
])
def test_attend_fp8_cascade_small(pkvlib, hq, hkv, prefix, suffixes):
    lens = [prefix + s for s in suffixes]
    b = make_batch(lens, [1] * len(lens), hq, hkv, seed=prefix + 3, device="cuda",
                   pool_factor=1.0, shared_prefix_tokens=prefix)
    out, expected = _cascade_fp8(b, prefix // 16, prefix, max_query_len=1)
    compare(out, expected, what=f"fp8 cascade {hq}/{hkv} prefix {prefix}")


def test_attend_fp8_cascade_with_prefill_chunk(pkvlib):
    """A shared prefix with decode rows, a short multi-row chunk (split-KV)
    and a long chunk (tensor-core prefill reading the prefix itself)."""
    prefix = 512
    b = make_batch([prefix + 30, prefix + 200, prefix + 9], [1, 40, 9], 32, 8, seed=79,
                   device="cuda", pool_factor=1.0, shared_prefix_tokens=prefix)
    out, expected = _cascade_fp8(b, prefix // 16, 79)
    compare(out, expected, what="fp8 cascade mixed")


def test_attend_fp8_close_to_bf16_attention_of_the_same_rows(pkvlib):
    """Same batch, bf16 pool vs the FP8 pool written from the same rows: the
    two results agree to the accuracy of E4M3 (a sanity check of scale
    handling, not a parity bar)."""
    b = workload(1, device="cuda")
    meta = to_device(b)
    kc16, vc16 = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc16, vc16)
    # encode the whole written bf16 pool as one batch of rows
    NB, Hkv = b.num_blocks, b.num_kv_heads
    rows_k = kc16.reshape(NB * Hkv * 16, 1, 128)
    rows_v = vc16.reshape(NB * Hkv * 16, 1, 128)
    slots = torch.arange(NB * Hkv * 16, dtype=torch.int64, device="cuda")
    flat = [torch.zeros(NB * Hkv * 16, 1, 16, 128, dtype=torch.uint8, device="cuda") for _ in range(2)] + \
           [torch.zeros(NB * Hkv * 16, 1, 16, dtype=torch.uint8, device="cuda") for _ in range(2)]
    pkv.write_fp8(rows_k, rows_v, slots * 16, *flat)
    kc8 = flat[0][:, 0, 0].reshape(NB, Hkv, 16, 128).contiguous()
    vc8 = flat[1][:, 0, 0].reshape(NB, Hkv, 16, 128).contiguous()
    ks8 = flat[2][:, 0, 0].reshape(NB, Hkv, 16).contiguous()
    vs8 = flat[3][:, 0, 0].reshape(NB, Hkv, 16).contiguous()
    o16 = pkv.attend(b.q, kc16, vc16, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale)
    o8 = pkv.attend_fp8(b.q, kc8, vc8, ks8, vs8, meta["block_tables"], meta["seq_lens"],
                        meta["query_start_loc"], b.scale)
    torch.cuda.synchronize()
    err = (o16.float() - o8.float()).abs()
    assert float(err.max()) < 0.15 and float(err.mean()) < 0.02


def test_attend_fp8_rejects_bad_arguments(pkvlib):
    b = workload(1, device="cuda")
    kc, vc, ks, vs = fp8_pools(b, 1)
    meta = to_device(b)
    lib = pkv.lib()
    desc = pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1])
    ws = torch.empty(pkv.workspace_size_fp8(desc, b.B, b.T, "cuda"), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(b.q)
    import ctypes
    P = pkv._ptr
    args = lambda ksp: (P(b.q), P(kc), P(vc), ksp, P(vs), P(meta["block_tables"]), P(meta["seq_lens"]),
                        P(meta["query_start_loc"]), b.B, b.T, 0, 0, ctypes.c_float(b.scale), P(out), P(ws),
                        ws.numel(), ctypes.byref(desc), pkv._stream(b.q.device, None))
    assert lib.pkv_attend_fp8(*args(ctypes.c_void_p(0))) == -1          # PKV_ERR_NULL
    assert lib.pkv_attend_fp8(*args(ctypes.c_void_p(ks.data_ptr() + 1))) == -2  # PKV_ERR_ALIGN
    assert lib.pkv_attend_fp8(*args(P(ks))) == 0
    short = ctypes.c_size_t(ws.numel() - 256)
    a = list(args(P(ks)))
    a[15] = short
    assert lib.pkv_attend_fp8(*a) == -5  # PKV_ERR_WORKSPACE
    torch.cuda.synchronize()


# Outputs of magnitude 2..3.875 (bf16 spacing 2^-6): the P of the FP8 paths
# (f16 in split-KV, bf16 in the tensor-core kernel) must not add a rounding
# of its own.  The pool's V codes and this step's new V rows both stand for
# such values.

@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 8), (8, 8)])
def test_attend_fp8_short_decode_rows_with_large_outputs(pkvlib, hq, hkv):
    lens = np.random.default_rng(hq + 1).integers(1, 25, size=768).tolist()
    b = large_value_rows(make_batch(lens, [1] * len(lens), hq, hkv, seed=520 + hq, device="cuda"), 620 + hq)
    _run(b, 720 + hq, v_values=b.v_cache, what=f"fp8 short rows, large outputs {hq}/{hkv}",
         cmp=compare_large_outputs)


@pytest.mark.parametrize("hq,hkv,chunks", [(32, 8, [300, 200]), (8, 8, [260])])
def test_attend_fp8_prefill_from_position_zero_with_large_outputs(pkvlib, hq, hkv, chunks):
    b = large_value_rows(make_batch(chunks + [40], chunks + [1], hq, hkv, seed=740 + sum(chunks),
                                    device="cuda"), 840 + hq)
    _run(b, 760 + hq, v_values=b.v_cache, what=f"fp8 prefill from 0, large outputs {hq}/{hkv}",
         cmp=compare_large_outputs)


def test_attend_fp8_prefill_bad_block_ids_are_flagged(pkvlib):
    """The FP8 prefill loaders stage pages by block id: ids inside the key
    window that are not pool pages are flagged and page 0 is staged instead;
    the other sequences' rows are unaffected."""
    b = make_batch([600, 300, 50], [200, 100, 1], 32, 8, seed=903, device="cuda")
    pools = fp8_pools(b, 904)
    meta = to_device(b)
    kc, vc, ks, vs = _gpu_write(b, pools, meta)
    meta["block_tables"][0, 3] = -5
    meta["block_tables"][0, 20] = b.num_blocks + 7
    pkv.get_last_error()
    out = pkv.attend_fp8(b.q, kc, vc, ks, vs, meta["block_tables"], meta["seq_lens"],
                         meta["query_start_loc"], b.scale, max_query_len=200)
    torch.cuda.synchronize()
    assert pkv.get_last_error() & pkv.STATUS_BAD_BLOCK
    ref = _oracle_write(b, pools)
    rows = list(range(200, b.T))
    expected = O.attend_fp8(bits(b.q), *ref, b.block_tables, b.seq_lens, b.query_start_loc, b.scale,
                            b.num_q_heads, b.num_kv_heads, b.page_size, rows=rows)
    compare(out, expected, rows=rows, what="fp8 rows beside bad block ids")


def test_attend_fp8_mixed_length_chunks(pkvlib):
    """FP8 pages: chunks of 9 to 200 query tokens over up to 3000 cached keys
    in one prefill launch, ragged last tiles of every length."""
    rng = np.random.default_rng(970)
    qlens = rng.integers(9, 200, size=20)
    lens = qlens + rng.integers(0, 3000, size=20)
    _run(make_batch(lens.tolist(), qlens.tolist(), 32, 8, seed=971, device="cuda"), 972,
         what="fp8 mixed-length chunks")
