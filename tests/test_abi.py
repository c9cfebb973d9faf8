"""The C ABI: every symbol include/pkv.h declares is exported, and argument
errors are rejected on the host before anything touches a GPU."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_pkv_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)


def test_header_declares_the_two_calls():
    names = declared_functions()
    assert "pkv_write" in names and "pkv_attend" in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(pkvlib):
    for name in declared_functions():
        assert hasattr(pkvlib, name), name


def test_binding_covers_every_symbol(pkvlib):
    assert set(declared_functions()) <= set(pkv._SIGS)


def _desc(**kw):
    d = dict(num_blocks=64, page_size=16, num_kv_heads=2, num_q_heads=8, head_dim=128,
             max_blocks_per_seq=16)
    d.update(kw)
    return pkv.Desc(**d)


FAKE = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced


def _write(lib, desc, **ptrs):
    p = dict(k_new=FAKE, v_new=FAKE, slots=FAKE, k_cache=FAKE, v_cache=FAKE)
    p.update(ptrs)
    return lib.pkv_write(p["k_new"], p["v_new"], p["slots"], 4, p["k_cache"], p["v_cache"],
                         ctypes.byref(desc), None)


def _attend(lib, desc, B=4, T=4, **ptrs):
    p = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, qsl=FAKE, out=FAKE, ws=FAKE)
    p.update(ptrs)
    return lib.pkv_attend(p["q"], p["kc"], p["vc"], p["bt"], p["sl"], p["qsl"], B, T, 0, 0, 0.1,
                          p["out"], p["ws"], 1 << 20, ctypes.byref(desc), None)


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=64), -3), (dict(page_size=32), -3), (dict(num_q_heads=6, num_kv_heads=4), -3),
    (dict(num_q_heads=24, num_kv_heads=8), -3), (dict(num_kv_heads=0), -3),
    (dict(num_blocks=0), -4), (dict(max_blocks_per_seq=0), -4),
])
def test_bad_geometry_rejected(pkvlib, bad, code):
    assert _write(pkvlib, _desc(**bad)) == code
    assert _attend(pkvlib, _desc(**bad)) == code
    n = ctypes.c_size_t(0)
    assert pkvlib.pkv_attend_workspace_size(ctypes.byref(_desc(**bad)), 4, 4, 0, ctypes.byref(n)) == code


def test_null_and_misaligned_pointers_rejected(pkvlib):
    d = _desc()
    assert _write(pkvlib, d, k_new=ctypes.c_void_p(0)) == -1
    assert _write(pkvlib, d, v_cache=ctypes.c_void_p(0)) == -1
    assert _write(pkvlib, d, k_cache=ctypes.c_void_p((1 << 20) + 8)) == -2
    assert _write(pkvlib, d, slots=ctypes.c_void_p((1 << 20) + 4)) == -2
    assert _attend(pkvlib, d, ws=ctypes.c_void_p(0)) == -1
    assert _attend(pkvlib, d, q=ctypes.c_void_p((1 << 20) + 2)) == -2
    assert _attend(pkvlib, d, ws=ctypes.c_void_p((1 << 20) + 128)) == -2
    assert _attend(pkvlib, d, B=-1) == -4
    assert pkvlib.pkv_write(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(d), None) == -4
    assert pkvlib.pkv_attend(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 0, 0, 0.1, FAKE, FAKE, 1 << 20,
                             None, None) == -1


def test_counts_out_of_range_rejected_before_any_device_work(pkvlib):
    """More sequences than PKV_MAX_SEQS, or a shared prefix longer than a
    block-table row, is a range error from every attention entry point and
    from the workspace queries, checked before a device is touched."""
    d = _desc()
    before = pkvlib.pkv_launch_count()
    assert _attend(pkvlib, d, B=2049, T=2049) == -4
    assert pkvlib.pkv_attend(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 0, d.max_blocks_per_seq + 1, 0.1,
                             FAKE, FAKE, 1 << 20, ctypes.byref(d), None) == -4
    for prefix, B in ((0, 2049), (d.max_blocks_per_seq + 1, 4)):
        assert pkvlib.pkv_attend_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, B, 0, prefix, 0.1,
                                     FAKE, FAKE, 1 << 20, ctypes.byref(d), None) == -4
        n = ctypes.c_size_t(0)
        assert pkvlib.pkv_attend_workspace_size(ctypes.byref(d), B, B, prefix, ctypes.byref(n)) == -4
        assert pkvlib.pkv_attend_fp8_workspace_size(ctypes.byref(d), B, B, prefix, ctypes.byref(n)) == -4
    assert pkvlib.pkv_launch_count() == before


def test_empty_calls_launch_nothing(pkvlib):
    d = _desc()
    before = pkvlib.pkv_launch_count()
    assert pkvlib.pkv_write(None, None, None, 0, None, None, ctypes.byref(d), None) == 0
    assert _attend(pkvlib, d, B=0, T=0) == 0
    assert pkvlib.pkv_launch_count() == before


def test_strerror_covers_every_code(pkvlib):
    for code in range(0, -11, -1):
        assert pkvlib.pkv_strerror(code) not in (None, b"unknown error")
    assert pkvlib.pkv_strerror(-99) == b"unknown error"


def test_trace_api_misuse(pkvlib):
    assert pkvlib.pkv_trace_detach() == -8
    assert pkvlib.pkv_trace_attach(None) == -1
    assert pkvlib.pkv_trace_create(0, ctypes.byref(ctypes.c_void_p())) == -4
