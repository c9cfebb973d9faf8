"""Seeded synthetic inputs for the paged-KV-cache hot path.

This module is the one thing the CUDA path and the float64 oracle share.  It
builds what a serving scheduler would hand to one step of a continuous batch
-- sequence lengths, query row offsets, per-sequence block tables over a
shuffled page pool, the slot of every new token -- plus the bf16 tensors
(queries, new K/V rows, the whole pre-filled page pool).  It holds none of the
method's arithmetic: no attention, no write, no merge.

Randomness: lengths, permutations and slots come from
``numpy.random.Generator(PCG64(seed))``; tensor values are N(0, 1) float32
from a ``torch.Generator`` seeded with the same number on the target device,
rounded to bf16 (round-to-nearest-even, torch ``.to(bfloat16)``).

The five named workloads follow the serving shapes they are named for
(Llama-3-8B-like heads: 32 query / 8 KV heads, head_dim 128, 16-token pages).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
PAGE_SIZE = 16

WORKLOADS = {
    1: "tiny paged decode: 4 seqs, L={17,64,100,255}, 8 q / 2 kv heads, 64-page pool",
    2: "Llama-3-8B-shaped decode layer: 64 seqs, L~U{512..4096}, 32 q / 8 kv heads, pool 1.25x need",
    3: "long-tail continuous batch: 256 decode seqs, L log-uniform 16..32768, 32 q / 8 kv heads",
    4: "prefix-shared decode: 128 seqs sharing 2048 prefix tokens, unique 64..256-token suffixes",
    5: "mixed step: 96 decode seqs L~U{256..8192} + prefill chunks of 512 over 1536 and 3584 cached",
}


@dataclass
class Batch:
    """One step of a continuous batch.  Host metadata is numpy; tensors torch."""

    num_q_heads: int
    num_kv_heads: int
    num_blocks: int
    seq_lens: np.ndarray          # [B] int32, includes this step's new tokens
    query_start_loc: np.ndarray   # [B+1] int32
    block_tables: np.ndarray      # [B, max_blocks] int32
    slot_mapping: np.ndarray      # [T] int64
    scale: float
    q: torch.Tensor = None        # [T, Hq, D] bf16
    k_new: torch.Tensor = None    # [T, Hkv, D] bf16
    v_new: torch.Tensor = None
    k_cache: torch.Tensor = None  # [NB, Hkv, P, D] bf16 (state before the write)
    v_cache: torch.Tensor = None
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    name: str = ""
    info: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc.astype(np.int64))


def _fill(shape, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def make_batch(seq_lens, q_lens, num_q_heads, num_kv_heads, seed, *,
               device="cpu", pool_factor=1.25, shared_prefix_tokens=0,
               extra_blocks=0, unused_table_value=None, name="custom",
               with_tensors=True, value_device=None):
    """Build a batch from per-sequence lengths.

    seq_lens[b] = tokens of sequence b after this step; q_lens[b] = new tokens
    (queries) this step, at positions seq_lens[b]-q_lens[b] .. seq_lens[b]-1.
    Pages are drawn from a shuffled pool of ceil(pool_factor * need) pages
    (+extra_blocks).  With shared_prefix_tokens > 0 (a multiple of the page
    size) every sequence's table starts with the same prefix pages, which are
    read-only: no new token of this step lands in them.
    Unused table entries hold ``unused_table_value`` (default: num_blocks,
    an out-of-range page id, so a read past a sequence's pages is visible).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    P = PAGE_SIZE
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = len(seq_lens)
    if np.any(q_lens > seq_lens) or np.any(q_lens < 0):
        raise ValueError("each q_len must be in [0, seq_len]")
    if shared_prefix_tokens % P:
        raise ValueError("shared prefix must be whole pages")
    n_pref = shared_prefix_tokens // P
    if n_pref and np.any(seq_lens - q_lens < shared_prefix_tokens):
        raise ValueError("new tokens may not land in shared prefix pages")
    pages_per_seq = (seq_lens + P - 1) // P
    own_pages = pages_per_seq - n_pref
    need = int(own_pages.sum()) + n_pref
    num_blocks = int(math.ceil(pool_factor * need)) + int(extra_blocks)
    perm = rng.permutation(num_blocks).astype(np.int64)
    max_blocks = int(pages_per_seq.max()) if B else 1
    fill = num_blocks if unused_table_value is None else int(unused_table_value)
    bt = np.full((B, max(max_blocks, 1)), fill, dtype=np.int64)
    cursor = 0
    prefix_pages = perm[:n_pref]
    cursor = n_pref
    for b in range(B):
        bt[b, :n_pref] = prefix_pages
        k = int(own_pages[b])
        bt[b, n_pref:n_pref + k] = perm[cursor:cursor + k]
        cursor += k
    qsl = np.zeros(B + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(q_lens)
    T = int(qsl[-1])
    slots = np.empty(T, dtype=np.int64)
    for b in range(B):
        L, n = int(seq_lens[b]), int(q_lens[b])
        pos = np.arange(L - n, L)
        slots[qsl[b]:qsl[b + 1]] = bt[b, pos // P] * P + pos % P
    batch = Batch(
        num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, num_blocks=num_blocks,
        seq_lens=seq_lens.astype(np.int32), query_start_loc=qsl.astype(np.int32),
        block_tables=bt.astype(np.int32), slot_mapping=slots,
        scale=float(np.float32(1.0 / math.sqrt(HEAD_DIM))), name=name,
    )
    batch.info = dict(seed=seed, pool_pages=num_blocks, pages_needed=need,
                      shared_prefix_pages=n_pref)
    if with_tensors:
        dev = torch.device(value_device or device)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        D = HEAD_DIM
        batch.k_cache = _fill((num_blocks, num_kv_heads, P, D), gen, dev)
        batch.v_cache = _fill((num_blocks, num_kv_heads, P, D), gen, dev)
        batch.q = _fill((T, num_q_heads, D), gen, dev)
        batch.k_new = _fill((T, num_kv_heads, D), gen, dev)
        batch.v_new = _fill((T, num_kv_heads, D), gen, dev)
        if torch.device(device) != dev:
            for name_ in ("k_cache", "v_cache", "q", "k_new", "v_new"):
                setattr(batch, name_, getattr(batch, name_).to(device))
    return batch


def workload(idx, *, device="cpu", with_tensors=True):
    """The five named workloads (see WORKLOADS), seeded with 1000 + idx."""
    seed = 1000 + idx
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    if idx == 1:
        lens = [17, 64, 100, 255]
        b = make_batch(lens, [1] * 4, 8, 2, seed, device=device, pool_factor=1.0,
                       extra_blocks=64 - 29, with_tensors=with_tensors)
    elif idx == 2:
        lens = rng.integers(512, 4096, size=64, endpoint=True)
        b = make_batch(lens, np.ones(64), 32, 8, seed, device=device,
                       with_tensors=with_tensors)
    elif idx == 3:
        u = rng.uniform(math.log(16), math.log(32768), size=256)
        lens = np.clip(np.round(np.exp(u)), 16, 32768).astype(np.int64)
        b = make_batch(lens, np.ones(256), 32, 8, seed, device=device, pool_factor=1.0,
                       with_tensors=with_tensors)
    elif idx == 4:
        suffix = rng.integers(64, 256, size=128, endpoint=True)
        b = make_batch(2048 + suffix, np.ones(128), 32, 8, seed, device=device,
                       pool_factor=1.0, shared_prefix_tokens=2048, with_tensors=with_tensors)
    elif idx == 5:
        dec = rng.integers(256, 8192, size=96, endpoint=True)
        lens = np.concatenate([dec, [1536 + 512, 3584 + 512]])
        qlens = np.concatenate([np.ones(96, dtype=np.int64), [512, 512]])
        b = make_batch(lens, qlens, 32, 8, seed, device=device, with_tensors=with_tensors)
    else:
        raise KeyError(idx)
    b.name = f"cfg{idx}"
    b.info["description"] = WORKLOADS[idx]
    return b


def large_value_rows(batch: Batch, seed: int, lo: float = 2.0, hi: float = 3.875):
    """Rewrite V (the pre-filled pool and this step's new rows) in place:
    every element gets a sign fixed per (kv head, dim) and a magnitude
    uniform in [lo, hi], rounded to bf16.  Any convex combination of such
    rows (an attention output) then has magnitude in [lo, hi]: with the
    defaults that is [2, 3.875], where bf16 values are 2^-6 apart, the
    hardest range for an absolute tolerance of 1e-2.  Values come from a
    torch.Generator seeded with ``seed`` on the batch's device."""
    dev = batch.v_cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    hkv, d = batch.num_kv_heads, batch.head_dim
    sign = torch.randint(0, 2, (hkv, d), generator=gen, device=dev).to(torch.float32) * 2 - 1

    def draw(shape, sgn):
        mag = lo + (hi - lo) * torch.rand(shape, generator=gen, device=dev, dtype=torch.float32)
        return (mag * sgn).to(torch.bfloat16)

    batch.v_cache = draw(tuple(batch.v_cache.shape), sign[None, :, None, :])
    batch.v_new = draw(tuple(batch.v_new.shape), sign[None, :, :])
    return batch


# Scale byte of the pre-filled FP8 pool: 2^(121 - 127) = 1/64.
FP8_FILL_SCALE_BYTE = 121


def fp8_pools(batch: Batch, seed: int, v_values: torch.Tensor = None):
    """A pre-filled FP8 page pool for ``batch``: E4M3 codes [NB, Hkv, P, D]
    (uint8) of N(0, 1) * 64 values (clipped to the format's +-448, which
    N(0, 1) reaches only beyond 7 sigma) and a constant scale byte
    FP8_FILL_SCALE_BYTE [NB, Hkv, P] (uint8), so the pool holds values close
    to N(0, 1).  Codes come from torch's float8_e4m3fn conversion with a
    torch.Generator seeded with ``seed``, on the batch's device.  With
    ``v_values`` (a pool-shaped tensor of magnitudes below 7) the V codes
    stand for those values times 64 instead.  No per-row scaling: that is
    the write step's arithmetic, done only by the write under test.
    Returns (k_codes, v_codes, k_scale, v_scale)."""
    dev = batch.q.device if batch.q is not None else torch.device("cpu")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    shape = (batch.num_blocks, batch.num_kv_heads, batch.page_size, batch.head_dim)
    out = []
    for i in range(2):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * 64.0
        if i == 1 and v_values is not None:
            x = v_values.to(device=dev, dtype=torch.float32) * 64.0
        out.append(x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
    sc = torch.full(shape[:3], FP8_FILL_SCALE_BYTE, dtype=torch.uint8, device=dev)
    return out[0], out[1], sc, sc.clone()


def kv_bytes(batch: Batch, unique: bool = True, fp8: bool = False) -> int:
    """Bytes of K+V rows a step must read: tokens < L of each sequence.

    unique=True counts a page shared by several block tables once (the bytes
    the method has to move); unique=False counts it once per reader.  fp8:
    rows of E4M3 codes plus one scale byte each.
    """
    P = batch.page_size
    row = 2 * batch.num_kv_heads * (batch.head_dim + 1 if fp8 else batch.head_dim * 2)
    if not unique:
        return int(batch.seq_lens.astype(np.int64).sum()) * row
    seen = {}
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for j in range((L + P - 1) // P):
            page = int(batch.block_tables[b, j])
            seen[page] = max(seen.get(page, 0), min(P, L - j * P))
    return sum(seen.values()) * row
