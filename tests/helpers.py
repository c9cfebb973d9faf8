"""Shared test helpers: bit views, oracle runs on a Batch, tolerance checks."""

import numpy as np
import torch

import oracle.pkv_oracle as O

# tolerance for attention outputs (bf16 result vs the float64 oracle): the
# bf16 rounding of an output of magnitude <= 4 is at most 8e-3
MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_device(batch, device="cuda"):
    """Metadata tensors of a workloads.Batch on the device."""
    dev = torch.device(device)
    return dict(
        seq_lens=torch.from_numpy(batch.seq_lens.astype(np.int32)).to(dev),
        query_start_loc=torch.from_numpy(batch.query_start_loc.astype(np.int32)).to(dev),
        block_tables=torch.from_numpy(batch.block_tables.astype(np.int32)).to(dev),
        slot_mapping=torch.from_numpy(batch.slot_mapping.astype(np.int64)).to(dev),
    )


def oracle_write(batch, slots=None):
    """Oracle write applied to the batch's initial pools (host uint16)."""
    s = batch.slot_mapping if slots is None else slots
    return O.write(bits(batch.k_new), bits(batch.v_new), s, bits(batch.k_cache),
                   bits(batch.v_cache), batch.page_size)


def oracle_attend(batch, k_pool, v_pool, rows=None, q=None):
    qq = bits(batch.q) if q is None else q
    return O.attend(qq, k_pool, v_pool, batch.block_tables, batch.seq_lens,
                    batch.query_start_loc, batch.scale, batch.num_q_heads,
                    batch.num_kv_heads, batch.page_size, rows=rows)


def compare(out_gpu: torch.Tensor, expected: np.ndarray, rows=None, what=""):
    """Max/mean abs error of GPU bf16 output vs float64 oracle on ``rows``."""
    got = O.bf16_to_f64(bits(out_gpu))
    if rows is not None:
        got, expected = got[rows], expected[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - expected)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Finite float64 values rounded to bf16 (through float32; ties to even),
    returned as float64."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def compare_large_outputs(out_gpu: torch.Tensor, expected: np.ndarray, rows=None, what=""):
    """Outputs of magnitude 2..4, where bf16 values are 2^-6 apart.  The max
    bar stays 1e-2.  No bf16 result can have a mean error below that of the
    exact result rounded to bf16 (about 2^-8 here, four times the 1e-3 bar
    set for N(0, 1) data), so the mean bar is that floor plus 2e-4."""
    got = O.bf16_to_f64(bits(out_gpu))
    if rows is not None:
        got, expected = got[rows], expected[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - expected)
    floor = float(np.abs(round_to_bf16(expected) - expected).mean())
    mx, mean = float(err.max()), float(err.mean())
    assert np.abs(expected).min() >= 1.99, f"{what}: outputs are not all large"
    assert mx <= MAX_ABS_TOL and mean <= floor + 2e-4, \
        f"{what}: max {mx:.3e} mean {mean:.3e} (rounding floor {floor:.3e})"
    return mx, mean
