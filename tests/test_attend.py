"""pkv_attend parity against the float64 oracle (max |err| <= 1e-2, mean <= 1e-3).

Small batches are compared on every output; the full-size named workloads on
all rows where the oracle is quick and on a sample of rows (shortest, longest,
first/last prefill rows, random) where it is not.
"""

import base64
import json
import os

import numpy as np
import pytest
import torch

import oracle.pkv_oracle as O
import paged_kv_cache_pkv_gb300 as pkv
from helpers import bits, compare, compare_large_outputs, oracle_attend, oracle_write, to_device
from workloads import large_value_rows, make_batch, workload

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def run_step(batch, meta=None, out=None):
    """pkv_write then pkv_attend on a fresh copy of the batch's pools."""
    meta = meta or to_device(batch)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    pkv.write(batch.k_new, batch.v_new, meta["slot_mapping"], kc, vc)
    out = pkv.attend(batch.q, kc, vc, meta["block_tables"], meta["seq_lens"],
                     meta["query_start_loc"], batch.scale, out=out)
    torch.cuda.synchronize()
    return out, kc, vc


def check_batch(batch, rows=None, what=""):
    out, kc, vc = run_step(batch)
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(batch)
    expected = oracle_attend(batch, k_ref, v_ref, rows=rows)
    return compare(out, expected, rows=rows, what=what or batch.name)


def test_golden_tiny_mixed(pkvlib):
    g = json.load(open(os.path.join(HERE, "golden", "tiny_mixed.json")))
    dec = lambda k, dt: np.frombuffer(base64.b64decode(g[k]), dtype=dt)
    Hq, Hkv, D, P, NB, T = g["num_q_heads"], g["num_kv_heads"], 128, 16, g["num_blocks"], g["T"]
    t16 = lambda k, shape: torch.from_numpy(dec(k, np.int16).reshape(shape).copy()).view(torch.bfloat16).cuda()
    q = t16("q", (T, Hq, D))[: g["num_query_rows"]].contiguous()
    kc, vc = t16("k_cache", (NB, Hkv, P, D)), t16("v_cache", (NB, Hkv, P, D))
    pkv.write(t16("k_new", (T, Hkv, D)), t16("v_new", (T, Hkv, D)),
              torch.tensor(g["slot_mapping"], dtype=torch.int64).cuda(), kc, vc)
    out = pkv.attend(q, kc, vc, torch.tensor(g["block_tables"], dtype=torch.int32).cuda(),
                     torch.tensor(g["seq_lens"], dtype=torch.int32).cuda(),
                     torch.tensor(g["query_start_loc"], dtype=torch.int32).cuda(), g["scale"])
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc).ravel(), dec("k_cache_after", np.uint16))
    assert np.array_equal(bits(vc).ravel(), dec("v_cache_after", np.uint16))
    expected = dec("out_f64", np.float64).reshape(T, Hq, D)[: g["num_query_rows"]]
    compare(out, expected, what="golden")


@pytest.mark.parametrize("idx", [1, 2, 4])
def test_named_workload_all_rows(pkvlib, idx):
    check_batch(workload(idx, device="cuda"))


def long_tail_rows(b, n=64, seed=0):
    """The ten longest rows of the long-tail batch (the widest splits), the
    shortest, and random others: ``n`` rows in all."""
    order = np.argsort(b.seq_lens, kind="stable")
    pick = set(order[-10:].tolist()) | {int(order[0])}
    rest = [r for r in range(b.B) if r not in pick]
    pick |= set(np.random.default_rng(seed).choice(rest, n - len(pick), replace=False).tolist())
    return sorted(pick)


def test_long_tail_rows(pkvlib):
    b = workload(3, device="cuda")
    check_batch(b, rows=long_tail_rows(b), what="cfg3 64 rows")


def test_mixed_step_all_rows(pkvlib):
    """Every one of the 1,120 rows: 96 decode rows on split-KV and both
    512-row chunks on the tensor-core pass running beside it."""
    b = workload(5, device="cuda")
    assert b.query_start_loc[-1] == 1120
    check_batch(b, what="cfg5 all rows")


@pytest.mark.parametrize("seed", range(6))
def test_random_small_batches(pkvlib, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 9))
    lens = rng.integers(1, 301, size=B)
    qlens = np.array([int(rng.integers(1, min(40, L) + 1)) if rng.random() < 0.4 else 1 for L in lens])
    hq, hkv = [(8, 2), (32, 8), (4, 4), (16, 2), (8, 4)][seed % 5]
    check_batch(make_batch(lens, qlens, hq, hkv, seed=seed, device="cuda"))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_group_sizes(pkvlib, G):
    hkv = 2
    check_batch(make_batch([33, 250, 16, 1], [1, 1, 16, 1], G * hkv, hkv, seed=40 + G, device="cuda"))


def test_zero_length_queries_and_idle_rows(pkvlib):
    """Sequences with no query this step produce nothing; rows past the last
    sequence's queries are left untouched."""
    b = make_batch([40, 17, 90, 5], [1, 0, 3, 0], 8, 2, seed=9, device="cuda")
    meta = to_device(b)
    q = torch.cat([b.q, b.q[:2]])  # two trailing rows owned by nobody
    out = torch.full_like(q, 7.0)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    pkv.attend(q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale, out=out)
    torch.cuda.synchronize()
    k_ref, v_ref = oracle_write(b)
    expected = oracle_attend(b, k_ref, v_ref)
    compare(out[: b.T], expected, what="zero-length")
    assert torch.all(out[b.T:] == 7.0)


def test_stale_nan_rows_do_not_leak(pkvlib):
    """Rows of a sequence's last page beyond its length hold NaN; they must
    not reach the output."""
    b = make_batch([17, 33, 250, 64], [1, 4, 1, 20], 8, 2, seed=10, device="cuda")
    kc, vc = b.k_cache, b.v_cache
    for bi in range(b.B):
        L = int(b.seq_lens[bi])
        last = int(b.block_tables[bi, (L - 1) // 16])
        if L % 16:
            kc[last, :, L % 16:, :] = float("nan")
            vc[last, :, L % 16:, :] = float("inf")
    check_batch(b, what="nan-stale")


def test_prefix_shared_identical_suffix_rows_agree(pkvlib):
    """Two sequences sharing prefix pages and with identical suffix content
    and query give the same output up to summation order (their split-KV
    partitions fall at different pages)."""
    b = make_batch([2048 + 40, 2048 + 40, 2048 + 77], [1, 1, 1], 32, 8, seed=11, device="cuda",
                   pool_factor=1.0, shared_prefix_tokens=2048)
    bt = b.block_tables
    for j in range(128, 131):  # copy seq 0's suffix pages into seq 1's
        b.k_cache[int(bt[1, j])] = b.k_cache[int(bt[0, j])]
        b.v_cache[int(bt[1, j])] = b.v_cache[int(bt[0, j])]
    b.k_new[1] = b.k_new[0]
    b.v_new[1] = b.v_new[0]
    b.q[1] = b.q[0]
    out, _, _ = run_step(b)
    diff = (out[0].double() - out[1].double()).abs().max().item()
    assert diff <= 2e-3, diff
    check_batch(b, what="prefix")


def test_bad_block_id_is_flagged_not_read(pkvlib):
    b = make_batch([100, 40], [1, 1], 8, 2, seed=12, device="cuda")
    meta = to_device(b)
    meta["block_tables"][0, 2] = b.num_blocks + 1000  # live entry out of the pool
    pkv.get_last_error()
    run_step(b, meta)
    assert pkv.get_last_error() & pkv.STATUS_BAD_BLOCK


def test_query_longer_than_sequence_is_flagged(pkvlib):
    b = make_batch([10, 40], [1, 1], 8, 2, seed=13, device="cuda")
    meta = to_device(b)
    meta["seq_lens"][0] = 0  # 1 query row but 0 tokens
    pkv.get_last_error()
    run_step(b, meta)
    assert pkv.get_last_error() & pkv.STATUS_BAD_QUERY


def test_most_sequences_per_call(pkvlib):
    """PKV_MAX_SEQS decode sequences in one call fill the plan's per-sequence
    arrays in shared memory: every row against the oracle; one more sequence
    is a range error.  1-64 keys per row: with only a few keys an output is
    close to one V row (|out| near 4 on this data)."""
    lens = np.random.default_rng(2048).integers(1, 65, size=2048).tolist()
    b = make_batch(lens, [1] * 2048, 8, 2, seed=2048, device="cuda")
    check_batch(b, what="2048 sequences")
    meta = to_device(b)
    bt = torch.cat([meta["block_tables"], meta["block_tables"][:1]])
    sl = torch.cat([meta["seq_lens"], meta["seq_lens"][:1]])
    qsl = torch.arange(2050, dtype=torch.int32, device="cuda")
    q = torch.cat([b.q, b.q[:1]])
    with pytest.raises(pkv.PkvError) as err:
        pkv.attend(q, b.k_cache, b.v_cache, bt, sl, qsl, b.scale)
    assert err.value.code == -4


def test_repeated_calls_reuse_workspace(pkvlib):
    b = workload(2, device="cuda")
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    ws = torch.empty(pkv.workspace_size(pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1]),
                                        b.B, b.T), dtype=torch.uint8, device="cuda")
    outs = [pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"],
                       b.scale, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_repeated_mixed_calls_reuse_workspace(pkvlib):
    """Back-to-back calls with a prefill chunk and long split-KV work on one
    workspace: a call's kernels must not overlap the previous call's merges."""
    b = make_batch([3000] * 40 + [300], [1] * 40 + [200], 32, 8, seed=91, device="cuda")
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    ws = torch.empty(pkv.workspace_size(pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1]),
                                        b.B, b.T), dtype=torch.uint8, device="cuda")
    outs = [pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"],
                       b.scale, workspace=ws) for _ in range(4)]
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    k_ref, v_ref = oracle_write(b)
    compare(outs[-1], oracle_attend(b, k_ref, v_ref), what="repeated mixed calls")


def _kernel_launches(batch, max_query_len):
    meta = to_device(batch)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    pkv.write(batch.k_new, batch.v_new, meta["slot_mapping"], kc, vc)
    tr = pkv.Trace(64)
    with tr:
        out = pkv.attend(batch.q, kc, vc, meta["block_tables"], meta["seq_lens"],
                         meta["query_start_loc"], batch.scale, max_query_len=max_query_len)
    torch.cuda.synchronize()
    counts = {k: tr.read(k)[1] for k in ("decode", "prefill")}
    tr.close()
    return counts, out, kc, vc


def test_long_chunks_run_on_the_tensor_core_kernel(pkvlib):
    b = make_batch([700, 300, 90], [200, 1, 90], 8, 2, seed=30, device="cuda")
    counts, out, _, _ = _kernel_launches(b, 0)
    assert counts == {"decode": 1, "prefill": 1}
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what="prefill full rows")
    # a bound at or below the split threshold routes every row through split-KV
    counts, out2, _, _ = _kernel_launches(b, 1)
    assert counts == {"decode": 1, "prefill": 0}
    compare(out2, oracle_attend(b, k_ref, v_ref), what="split-KV all rows")


@pytest.mark.parametrize("hq,hkv,L,n", [(32, 8, 1100, 130), (16, 2, 257, 257), (8, 8, 640, 300),
                                        (32, 2, 129, 33), (64, 4, 3000, 17), (32, 8, 2000, 100),
                                        (16, 8, 700, 200)])
def test_prefill_chunks_all_rows(pkvlib, hq, hkv, L, n):
    """Chunks spanning several 128-key tiles with ragged ends, every row."""
    b = make_batch([L, 40], [n, 1], hq, hkv, seed=L + n, device="cuda")
    counts, out, _, _ = _kernel_launches(b, n)
    assert counts["prefill"] == 1
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what=f"prefill {hq}/{hkv} L={L} n={n}")


def test_prefill_chunk_over_a_long_context(pkvlib):
    """A 40-token chunk at the end of a 16,384-token sequence: its query
    group runs 128 K/V tiles, so the tile buffers and their barriers wrap
    their phases many times.  Every row against the oracle."""
    b = make_batch([16384, 300], [40, 1], 32, 8, seed=990, device="cuda")
    counts, out, _, _ = _kernel_launches(b, 40)
    assert counts["prefill"] == 1
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what="prefill over 16k keys")


def test_prefill_chunks_of_several_sequences(pkvlib):
    """Several prefill chunks in one step: query groups of two Q tiles per CTA,
    a last group with one tile or with a partial second tile, next to decode rows."""
    b = make_batch([2000, 1500, 64, 700, 333], [300, 77, 1, 36, 33], 32, 8, seed=77, device="cuda")
    counts, out, _, _ = _kernel_launches(b, 300)
    assert counts["prefill"] == 1
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what="several prefill chunks")


@pytest.mark.parametrize("lens,qlens", [
    ([3000] * 40 + [300], [1] * 40 + [200]),  # long split-KV work, short prefill chunk
    ([2048, 64], [512, 1]),                   # long prefill chunk, short split-KV work
    ([700, 500], [300, 200]),                 # prefill chunks only
])
def test_mixed_step_result_is_stream_ordered(pkvlib, lens, qlens):
    """A copy ordered on the stream right after pkv_attend (no device-wide
    synchronisation) reads the complete output, whichever of the split-KV
    kernel and the prefill pass finishes last."""
    b = make_batch(lens, qlens, 32, 8, seed=sum(lens), device="cuda")
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    out = torch.full_like(b.q, float("nan"))
    torch.cuda.synchronize()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
               out=out)
    host = out.cpu()  # stream-ordered copy
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare(host, oracle_attend(b, k_ref, v_ref), what=f"stream-ordered read {len(lens)} rows")


def _cascade(batch, prefix_pages, max_query_len=0):
    meta = to_device(batch)
    kc, vc = batch.k_cache.clone(), batch.v_cache.clone()
    pkv.write(batch.k_new, batch.v_new, meta["slot_mapping"], kc, vc)
    out = pkv.attend(batch.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"],
                     batch.scale, max_query_len=max_query_len, shared_prefix_pages=prefix_pages)
    torch.cuda.synchronize()
    return out


def test_cascade_prefix_shared_workload(pkvlib):
    """Config 4: 128 sequences on one 2048-token prefix, cascade vs oracle."""
    b = workload(4, device="cuda")
    out = _cascade(b, b.info["shared_prefix_pages"], max_query_len=1)
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what="cascade cfg4")


@pytest.mark.parametrize("hq,hkv,prefix,suffixes", [
    (32, 8, 80, [1, 17, 100, 16]),        # prefix of 5 pages: one partial key tile
    (16, 2, 1600, [3, 250, 33]),          # several key chunks of the prefix
    (8, 8, 256, [40, 1, 2]),              # one query head per kv head
    (64, 8, 512, [70, 5]),                # 8 query heads per kv head (two head groups)
    (8, 4, 16, [1, 2, 3, 4, 5]),          # one-page prefix, tiny suffixes
])
def test_cascade_small(pkvlib, hq, hkv, prefix, suffixes):
    lens = [prefix + s for s in suffixes]
    b = make_batch(lens, [1] * len(lens), hq, hkv, seed=prefix + len(suffixes), device="cuda",
                   pool_factor=1.0, shared_prefix_tokens=prefix)
    out = _cascade(b, prefix // 16, max_query_len=1)
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what=f"cascade {hq}/{hkv} prefix {prefix}")


def test_cascade_with_prefill_chunk_and_speculative_rows(pkvlib):
    """A shared prefix with decode rows, short multi-row chunks (split-KV) and
    a long chunk (tensor-core prefill, which reads the prefix itself)."""
    prefix = 512
    b = make_batch([prefix + 30, prefix + 200, prefix + 64, prefix + 9], [1, 40, 3, 9], 32, 8, seed=77,
                   device="cuda", pool_factor=1.0, shared_prefix_tokens=prefix)
    out = _cascade(b, prefix // 16)
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what="cascade mixed")


def test_cascade_row_without_own_key_is_flagged(pkvlib):
    b = make_batch([160, 200], [1, 1], 8, 2, seed=78, device="cuda", pool_factor=1.0,
                   shared_prefix_tokens=144)
    pkv.get_last_error()
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    # claim a 10-page prefix: sequence 0 (160 tokens) has no key past it
    pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
               max_query_len=1, shared_prefix_pages=10)
    assert pkv.get_last_error() & pkv.STATUS_BAD_QUERY


# Outputs of magnitude 2..3.875, where bf16 values are 2^-6 apart: the output
# rounding alone may cost 7.8e-3 of the 1e-2 budget, so P must not add a
# rounding of its own (one bf16 rounding of P moves an output by up to 2^-8
# of the V rows it weighs).  Rows with few keys have the least averaging.

@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 8), (8, 8), (64, 8)])
def test_short_decode_rows_with_large_outputs(pkvlib, hq, hkv):
    """Decode rows over 1-24 keys, every output element in [2, 3.875] in
    magnitude; query-head groups of 4, 2 and 1 (the page product's
    remainder columns sit differently for each) and 8 (two groups)."""
    lens = np.random.default_rng(hq).integers(1, 25, size=768).tolist()
    b = large_value_rows(make_batch(lens, [1] * len(lens), hq, hkv, seed=500 + hq, device="cuda"), 600 + hq)
    out, _, _ = run_step(b)
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare_large_outputs(out, oracle_attend(b, k_ref, v_ref), what=f"short rows, large outputs {hq}/{hkv}")


@pytest.mark.parametrize("hq,hkv,chunks", [(32, 8, [300, 200]), (8, 8, [260]), (16, 2, [129, 64])])
def test_prefill_from_position_zero_with_large_outputs(pkvlib, hq, hkv, chunks):
    """Chunks that start at position 0 (L = n: query j sees keys 0..j, so the
    first rows see one, two, three keys) on the tensor-core kernel, with
    every output element in [2, 3.875] in magnitude, next to a decode row."""
    lens = chunks + [40]
    b = large_value_rows(make_batch(lens, chunks + [1], hq, hkv, seed=700 + sum(chunks), device="cuda"),
                         800 + hq)
    counts, out, _, _ = _kernel_launches(b, max(chunks))
    assert counts["prefill"] == 1
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare_large_outputs(out, oracle_attend(b, k_ref, v_ref), what=f"prefill from 0, large outputs {hq}/{hkv}")


def test_prefill_bad_block_ids_are_flagged(pkvlib):
    """Table entries inside a prefill chunk's key window that are not pool
    pages (negative, and past the pool) are flagged, and page 0 is read in
    their place; the other sequences' rows are unaffected."""
    b = make_batch([600, 300, 50], [200, 100, 1], 32, 8, seed=901, device="cuda")
    meta = to_device(b)
    meta["block_tables"][0, 3] = -5
    meta["block_tables"][0, 20] = b.num_blocks + 7
    pkv.get_last_error()
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    tr = pkv.Trace(16)
    with tr:
        out = pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"],
                         b.scale, max_query_len=200)
    torch.cuda.synchronize()
    assert tr.read("prefill")[1] == 1
    tr.close()
    assert pkv.get_last_error() & pkv.STATUS_BAD_BLOCK
    k_ref, v_ref = oracle_write(b)
    rows = list(range(200, b.T))  # sequences 1 and 2
    compare(out, oracle_attend(b, k_ref, v_ref, rows=rows), rows=rows, what="rows beside bad block ids")


def test_cascade_bad_prefix_block_id_is_flagged(pkvlib):
    """A negative id among the shared prefix pages reaches the prefix pass's
    loaders, which flag it."""
    b = make_batch([512 + 30, 512 + 9], [1, 1], 32, 8, seed=902, device="cuda", pool_factor=1.0,
                   shared_prefix_tokens=512)
    meta = to_device(b)
    meta["block_tables"][:, 5] = -1
    pkv.get_last_error()
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
               max_query_len=1, shared_prefix_pages=32)
    torch.cuda.synchronize()
    assert pkv.get_last_error() & pkv.STATUS_BAD_BLOCK


@pytest.mark.parametrize("seed", [0, 1])
def test_mixed_length_chunks_beside_decode_rows(pkvlib, seed):
    """Two dozen chunks of 9 to 200 query tokens over up to 3000 cached keys,
    every fifth row a decode row: query groups of every length and ragged
    last tiles in one prefill launch beside split-KV.  Every row against the
    oracle; three calls on one workspace give the same bits."""
    rng = np.random.default_rng(950 + seed)
    B = 24
    qlens = rng.integers(9, 200, size=B)
    lens = qlens + rng.integers(0, 3000, size=B)
    qlens[::5] = 1  # decode rows beside them
    b = make_batch(lens.tolist(), qlens.tolist(), 32, 8, seed=960 + seed, device="cuda")
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    ws = torch.empty(pkv.workspace_size(pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1]), b.B, b.T),
                     dtype=torch.uint8, device="cuda")
    outs = [pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
                       workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    k_ref, v_ref = oracle_write(b)
    compare(outs[0], oracle_attend(b, k_ref, v_ref), what=f"mixed-length chunks {seed}")
