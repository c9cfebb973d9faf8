"""Bounded waits: when one runs out, the kernel flags PKV_STATUS_TIMEOUT, lets
its own copies and MMAs land, frees its TMEM and returns, and the device stays
usable.

Two test builds of the library with a wait limit of 2 ms, compiled beside the
main one and loaded next to it (each keeps its own status word), each with a
wait on something that nothing completes:
  * the first page copy of every split-KV warp and the Q tiles of every
    prefill CTA are armed on their barriers but never issued: split-KV warps,
    the prefill pass's MMA, softmax and loader warps (bf16 pages and the FP8
    loaders that widen pages) all see waits run out, drain what they did
    issue, free TMEM and return;
  * the arrival counters are left unstamped: every arrival of a split
    (row, head group) waits for the stamp until the limit.
After each, a normal call of the main library on the same stream must still
match the oracle.  No wait is unbounded, so nothing here can hang the GPU.
"""

import ctypes
import os

import pytest
import torch

import paged_kv_cache_pkv_gb300 as pkv
from paged_kv_cache_pkv_gb300 import build as pkv_build
from helpers import compare, oracle_attend, oracle_write, to_device
from workloads import fp8_pools, make_batch, workload

pytestmark = pytest.mark.gpu

_BUILD = os.path.join(os.path.dirname(pkv.__file__), "_build")


def _test_build(name, flags):
    path = pkv_build.build(extra_flags=flags, lib_path=os.path.join(_BUILD, f"libpkv_{name}.so"),
                           obj_dir=os.path.join(_BUILD, name))
    return pkv.open_library(path)


@pytest.fixture(scope="module")
def dropped_copy_lib(pkvlib):
    return _test_build("dropcopy", ["-DPKV_WAIT_LIMIT_NS=2000000ull", "-DPKV_TEST_DROP_FIRST_COPY"])


@pytest.fixture(scope="module")
def unstamped_lib(pkvlib):
    return _test_build("nostamp", ["-DPKV_WAIT_LIMIT_NS=2000000ull", "-DPKV_TEST_NO_EPOCH_STAMP"])


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _flags(lib):
    f = ctypes.c_uint32(0)
    assert lib.pkv_get_last_error(_stream(), ctypes.byref(f)) == 0
    return f.value


def _attend_with(lib, b, meta, kc, vc, max_query_len=0, fp8_scales=None):
    """pkv_attend (or pkv_attend_fp8) of ``lib`` into a NaN-filled output,
    with a zero-filled workspace of the size that build asks for."""
    desc = pkv.make_desc(kc, b.num_q_heads, b.block_tables.shape[1])
    need = ctypes.c_size_t(0)
    size_fn = lib.pkv_attend_fp8_workspace_size if fp8_scales else lib.pkv_attend_workspace_size
    assert size_fn(ctypes.byref(desc), b.B, b.T, 0, ctypes.byref(need)) == 0
    ws = torch.zeros(max(need.value, 256), dtype=torch.uint8, device="cuda")
    out = torch.full_like(b.q, float("nan"))
    common = (_p(meta["block_tables"]), _p(meta["seq_lens"]), _p(meta["query_start_loc"]), b.B, b.T,
              max_query_len, 0, b.scale, _p(out), _p(ws), ws.numel(), ctypes.byref(desc), _stream())
    if fp8_scales:
        rc = lib.pkv_attend_fp8(_p(b.q), _p(kc), _p(vc), _p(fp8_scales[0]), _p(fp8_scales[1]), *common)
    else:
        rc = lib.pkv_attend(_p(b.q), _p(kc), _p(vc), *common)
    assert rc == 0
    torch.cuda.synchronize()
    return out


def _main_library_still_correct(b, meta, kc, vc, max_query_len=0):
    pkv.get_last_error()
    out = pkv.attend(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], meta["query_start_loc"],
                     b.scale, max_query_len=max_query_len)
    torch.cuda.synchronize()
    assert pkv.get_last_error() == 0
    k_ref, v_ref = oracle_write(b)
    compare(out, oracle_attend(b, k_ref, v_ref), what=f"{b.name} after a timed-out call")


def _written(b):
    meta = to_device(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    pkv.write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc)
    return meta, kc, vc


@pytest.mark.parametrize("batch", ["decode", "mixed"])
def test_dropped_copy_waits_run_out_and_return(dropped_copy_lib, batch):
    torch.cuda.set_device(0)
    if batch == "decode":
        b, mql = workload(2, device="cuda"), 1
    else:  # split-KV first, the tensor-core prefill pass behind it
        b, mql = make_batch([2048, 1000, 300, 64], [512, 200, 1, 1], 32, 8, seed=950, device="cuda"), 512
    meta, kc, vc = _written(b)
    _flags(dropped_copy_lib)
    out = _attend_with(dropped_copy_lib, b, meta, kc, vc, max_query_len=mql)
    assert _flags(dropped_copy_lib) & pkv.STATUS_TIMEOUT
    assert torch.isnan(out.float()).any()  # rows whose first page never came stay unwritten
    _main_library_still_correct(b, meta, kc, vc, max_query_len=mql)


def test_dropped_copy_waits_run_out_in_the_fp8_loaders(dropped_copy_lib):
    torch.cuda.set_device(0)
    b = make_batch([1500, 700, 90], [300, 1, 1], 32, 8, seed=951, device="cuda")
    meta = to_device(b)
    kc, vc, ks, vs = (t.clone() for t in fp8_pools(b, 952))
    pkv.write_fp8(b.k_new, b.v_new, meta["slot_mapping"], kc, vc, ks, vs)
    _flags(dropped_copy_lib)
    _attend_with(dropped_copy_lib, b, meta, kc, vc, max_query_len=300, fp8_scales=(ks, vs))
    assert _flags(dropped_copy_lib) & pkv.STATUS_TIMEOUT
    meta2, kc2, vc2 = _written(b)
    _main_library_still_correct(b, meta2, kc2, vc2, max_query_len=300)


def test_unstamped_arrival_counters_time_out(unstamped_lib):
    """Eight 4096-token rows: every (row, head group) is split over many
    warps, so every one of them waits for a stamp that never comes; rows stay
    unwritten (NaN) and the call returns."""
    torch.cuda.set_device(0)
    b = make_batch([4096] * 8, [1] * 8, 32, 8, seed=953, device="cuda")
    meta, kc, vc = _written(b)
    _flags(unstamped_lib)
    out = _attend_with(unstamped_lib, b, meta, kc, vc, max_query_len=1)
    assert _flags(unstamped_lib) & pkv.STATUS_TIMEOUT
    assert torch.isnan(out.float()).all()  # no merge ever ran
    _main_library_still_correct(b, meta, kc, vc, max_query_len=1)
