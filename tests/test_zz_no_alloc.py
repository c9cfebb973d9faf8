"""pkv_attend_static: attention for callers that cannot allocate device memory.

Such callers -- code inside a host program that owns all device memory and
forbids allocation after start-up, or a C caller holding only pointers it was
given -- cannot create the workspace pkv_attend needs.  pkv_attend_static uses
a fixed scratch array inside the library instead.  This test calls it through
the C ABI twice in a row and checks that both results equal, bit for bit,
those of pkv_attend with a caller workspace (the kernels are deterministic),
and that they meet the attention tolerance against the float64 oracle; one
batch uses the shared-prefix cascade, whose prefix records also live in the
fixed array.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_pkv_gb300 as pkv
from helpers import compare, oracle_attend, oracle_write, to_device
from workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def _static_call(lib, b, meta, kc, vc, out, max_query_len=0, prefix_pages=0):
    desc = pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_attend_static(
        ctypes.c_void_p(b.q.data_ptr()), ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(meta["block_tables"].data_ptr()), ctypes.c_void_p(meta["seq_lens"].data_ptr()),
        ctypes.c_void_p(meta["query_start_loc"].data_ptr()), b.B, b.T, max_query_len, prefix_pages, b.scale,
        ctypes.c_void_p(out.data_ptr()), ctypes.byref(desc), stream)


@pytest.mark.parametrize("batch", ["llama8b_decode", "mixed_small", "shared_prefix"])
def test_static_scratch_matches_workspace_entry_point(pkvlib, batch):
    torch.cuda.set_device(0)
    mql, prefix_pages = 0, 0
    if batch == "llama8b_decode":
        b = workload(2, device="cuda")
    elif batch == "mixed_small":
        b = make_batch([33, 250, 16, 1, 700], [1, 1, 16, 1, 40], 32, 8, seed=3, device="cuda")
    else:  # 24 sequences on one 512-token prefix: cascade records in the fixed array
        suffixes = np.random.default_rng(4).integers(1, 200, size=24)
        b = make_batch((512 + suffixes).tolist(), [1] * 24, 32, 8, seed=4, device="cuda", pool_factor=1.0,
                       shared_prefix_tokens=512)
        mql, prefix_pages = 1, 32
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    ref = pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"], b.scale,
                     max_query_len=mql, shared_prefix_pages=prefix_pages)
    outs = []
    for _ in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert _static_call(pkvlib, b, meta, kc, vc, out, mql, prefix_pages) == 0
        outs.append(out)
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    for out in outs:
        assert torch.equal(out, ref)
    k_ref, v_ref = oracle_write(b)
    compare(outs[-1], oracle_attend(b, k_ref, v_ref), what=f"pkv_attend_static {batch}")


def test_static_scratch_rejects_oversized_batch(pkvlib):
    torch.cuda.set_device(0)
    desc = pkv.Desc(1024, 16, 8, 32, 128, 4)
    need = ctypes.c_size_t(0)
    T = 1 << 20  # per-row plan arrays alone exceed the fixed scratch
    assert pkvlib.pkv_attend_workspace_size(ctypes.byref(desc), 4, T, 0, ctypes.byref(need)) == 0
    assert need.value > (16 << 20)
    fake = ctypes.c_void_p(1 << 20)
    before = pkvlib.pkv_launch_count()
    assert pkvlib.pkv_attend_static(fake, fake, fake, fake, fake, fake, 4, T, 0, 0, 0.1, fake,
                                    ctypes.byref(desc), None) == -9
    assert pkvlib.pkv_launch_count() == before
