"""Python binding of libpkv -- the paged-KV-cache hot path for GB300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
shared library has not been built, importing works but every call raises
``PkvUnavailable``: there is no fallback.

    import paged_kv_cache_pkv_gb300 as pkv
    pkv.write(k_new, v_new, slot_mapping, k_cache, v_cache)
    out = pkv.attend(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale)
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PkvError", "PkvUnavailable", "lib", "open_library", "library_path", "Desc", "write", "attend",
    "workspace_size", "get_last_error", "launch_count", "Trace", "PagePool", "KERNELS",
    "export_pages", "import_pages", "write_fp8", "attend_fp8", "workspace_size_fp8",
    "STATUS_BAD_SLOT", "STATUS_BAD_BLOCK", "STATUS_BAD_QUERY", "STATUS_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.environ.get("PKV_LIBRARY", os.path.join(_HERE, "libpkv.so"))

STATUS_BAD_SLOT, STATUS_BAD_BLOCK, STATUS_BAD_QUERY, STATUS_TIMEOUT = 0x1, 0x2, 0x4, 0x8
KERNELS = {"write": 0, "plan": 1, "decode": 2, "merge": 3, "prefill": 4}


class PkvError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = _lib.pkv_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{what}: {msg} (code {code})" if what else f"{msg} (code {code})")


class PkvUnavailable(RuntimeError):
    pass


class Desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "pkv_write": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, ctypes.POINTER(Desc), _vp]),
    "pkv_attend_workspace_size": (ctypes.c_int, [ctypes.POINTER(Desc), _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "pkv_attend": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_float,
                                  _vp, _vp, _sz, ctypes.POINTER(Desc), _vp]),
    "pkv_attend_static": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                         ctypes.c_float, _vp, ctypes.POINTER(Desc), _vp]),
    "pkv_write_fp8": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, ctypes.POINTER(Desc), _vp]),
    "pkv_attend_fp8_workspace_size": (ctypes.c_int, [ctypes.POINTER(Desc), _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "pkv_attend_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_float,
                                      _vp, _vp, _sz, ctypes.POINTER(Desc), _vp]),
    "pkv_get_last_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "pkv_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_launch_count": (ctypes.c_uint64, []),
    "pkv_trace_create": (ctypes.c_int, [_i32, ctypes.POINTER(_vp)]),
    "pkv_trace_attach": (ctypes.c_int, [_vp]),
    "pkv_trace_detach": (ctypes.c_int, []),
    "pkv_trace_read": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64)]),
    "pkv_trace_reset": (ctypes.c_int, [_vp]),
    "pkv_trace_destroy": (ctypes.c_int, [_vp]),
    "pkv_export_pages": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, ctypes.POINTER(Desc), _vp]),
    "pkv_import_pages": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, ctypes.POINTER(Desc), _vp]),
    "pkv_pool_create": (ctypes.c_int, [_i32, ctypes.POINTER(_vp)]),
    "pkv_pool_destroy": (ctypes.c_int, [_vp]),
    "pkv_pool_alloc": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i32)]),
    "pkv_pool_retain": (ctypes.c_int, [_vp, ctypes.POINTER(_i32), _i32]),
    "pkv_pool_release": (ctypes.c_int, [_vp, ctypes.POINTER(_i32), _i32]),
    "pkv_pool_refcount": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i32)]),
    "pkv_pool_usage": (ctypes.c_int, [_vp, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "pkv_pool_make_writable": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, ctypes.POINTER(Desc), _vp,
                                              ctypes.POINTER(_i32)]),
}

_lib = None


def open_library(path):
    """A ctypes handle of a build of the library at ``path``, with every
    entry point's signature declared.  Each build loaded this way keeps its
    own device status word, launch count and caches."""
    if not os.path.exists(path):
        raise PkvUnavailable(
            f"{path} is missing: build it with "
            "`python -m paged_kv_cache_pkv_gb300.build` (nvcc, sm_103a)")
    handle = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(handle, name)
        fn.restype, fn.argtypes = res, args
    return handle


def lib():
    """The loaded shared library (raises PkvUnavailable if it is not built)."""
    global _lib
    if _lib is None:
        _lib = open_library(library_path)
    return _lib


def _check(code, what):
    if code != 0:
        raise PkvError(code, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")


def make_desc(k_cache, num_q_heads, max_blocks_per_seq):
    nb, hkv, p, d = k_cache.shape
    return Desc(nb, p, hkv, num_q_heads, d, max_blocks_per_seq)


def write(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """Scatter new K/V rows [T, Hkv, D] into the pools [NB, Hkv, P, D] at
    ``slot_mapping`` (int64 [T]; negative = skip).  In place, stream-ordered."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    if k_cache.shape != v_cache.shape or k_new.shape != v_new.shape or k_cache.dim() != 4:
        raise ValueError("k/v shapes disagree")
    T = k_new.shape[0]
    if slot_mapping.shape[0] != T or k_new.shape[1:] != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k_new must be [T, Hkv, D] matching the pool and slot_mapping")
    desc = make_desc(k_cache, k_cache.shape[1], 1)
    with torch.cuda.device(k_cache.device):
        _check(lib().pkv_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(k_cache),
                               _ptr(v_cache), ctypes.byref(desc), _stream(k_cache.device, stream)),
               "pkv_write")


def workspace_size(desc, num_seqs, num_tokens, device=None, shared_prefix_pages=0):
    n = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(lib().pkv_attend_workspace_size(ctypes.byref(desc), num_seqs, num_tokens,
                                               int(shared_prefix_pages), ctypes.byref(n)),
               "pkv_attend_workspace_size")
    return n.value


def attend(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out=None,
           workspace=None, stream=None, max_query_len=0, shared_prefix_pages=0):
    """Paged GQA attention of one continuous batch; returns ``out`` [T, Hq, D].

    ``workspace`` (uint8 CUDA tensor) may be passed to avoid an allocation by
    PyTorch's caching allocator on every call.  ``max_query_len`` is an
    optional host-side upper bound on query rows per sequence (0 = unknown);
    it only selects kernels, never results.  ``shared_prefix_pages`` > 0 says
    the first that many block-table entries of every row are the same pages
    (a common prefix), attended once for all rows (cascade)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T, Hq, D = q.shape
    B = seq_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("seq_lens [B], query_start_loc [B+1] and block_tables [B, M] disagree")
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("k_cache/v_cache/q shapes disagree")
    desc = make_desc(k_cache, Hq, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    need = workspace_size(desc, B, T, q.device, shared_prefix_pages)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    else:
        _need(workspace, "workspace", torch.uint8)
        if workspace.numel() < need:
            raise ValueError(f"workspace needs {need} bytes, got {workspace.numel()}")
    with torch.cuda.device(q.device):
        _check(lib().pkv_attend(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
                                _ptr(query_start_loc), B, T, int(max_query_len), int(shared_prefix_pages),
                                float(scale), _ptr(out),
                                _ptr(workspace), workspace.numel(), ctypes.byref(desc),
                                _stream(q.device, stream)),
               "pkv_attend")
    return out


def _need_fp8_pool(k_cache, v_cache, k_scale, v_scale):
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, 4)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.uint8, 3)
    if k_cache.shape != v_cache.shape or k_scale.shape != v_scale.shape or \
            tuple(k_scale.shape) != tuple(k_cache.shape[:3]):
        raise ValueError("FP8 pools must be codes [NB, Hkv, P, D] and scales [NB, Hkv, P]")


def write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """pkv_write into FP8 pages: new bf16 rows [T, Hkv, D] are encoded as E4M3
    codes (uint8 pools [NB, Hkv, P, D]) with one power-of-two scale byte per
    row (uint8 [NB, Hkv, P]).  In place, stream-ordered."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    T = k_new.shape[0]
    if k_new.shape != v_new.shape or slot_mapping.shape[0] != T or \
            k_new.shape[1:] != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k_new must be [T, Hkv, D] matching the pool and slot_mapping")
    desc = make_desc(k_cache, k_cache.shape[1], 1)
    with torch.cuda.device(k_cache.device):
        _check(lib().pkv_write_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(k_cache),
                                   _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), ctypes.byref(desc),
                                   _stream(k_cache.device, stream)),
               "pkv_write_fp8")


def workspace_size_fp8(desc, num_seqs, num_tokens, device=None, shared_prefix_pages=0):
    """Workspace bytes attend_fp8 needs for a batch of this size."""
    n = _sz(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(lib().pkv_attend_fp8_workspace_size(ctypes.byref(desc), int(num_seqs), int(num_tokens),
                                                   int(shared_prefix_pages), ctypes.byref(n)),
               "pkv_attend_fp8_workspace_size")
    return n.value


def attend_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, query_start_loc, scale,
               out=None, workspace=None, stream=None, max_query_len=0, shared_prefix_pages=0):
    """attend() over FP8 pages (codes and per-row scale bytes as written by
    write_fp8): long query chunks on the tensor-core prefill kernel, the rest
    on split-KV; max_query_len and shared_prefix_pages as in attend()."""
    _need(q, "q", torch.bfloat16, 3)
    _need_fp8_pool(k_cache, v_cache, k_scale, v_scale)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    T, Hq, D = q.shape
    B = seq_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("seq_lens [B], query_start_loc [B+1] and block_tables [B, M] disagree")
    if k_cache.shape[3] != D:
        raise ValueError("k_cache/q shapes disagree")
    desc = make_desc(k_cache, Hq, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    need = workspace_size_fp8(desc, B, T, q.device, shared_prefix_pages)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    else:
        _need(workspace, "workspace", torch.uint8)
        if workspace.numel() < need:
            raise ValueError(f"workspace needs {need} bytes, got {workspace.numel()}")
    with torch.cuda.device(q.device):
        _check(lib().pkv_attend_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(block_tables), _ptr(seq_lens), _ptr(query_start_loc), B, T,
                                    int(max_query_len), int(shared_prefix_pages), float(scale), _ptr(out),
                                    _ptr(workspace), workspace.numel(), ctypes.byref(desc),
                                    _stream(q.device, stream)),
               "pkv_attend_fp8")
    return out


def export_pages(k_cache, v_cache, pages, out=None, stream=None):
    """Copy whole pages into a contiguous buffer [n, 2, Hkv, 16, 128] bf16
    (device or pinned host tensor); returns it."""
    _need(pages, "pages", torch.int32, 1)
    n = pages.shape[0]
    if out is None:
        out = torch.empty((n, 2) + tuple(k_cache.shape[1:]), dtype=torch.bfloat16, device=k_cache.device)
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.numel() != n * 2 * k_cache[0].numel():
        raise ValueError("out must be a contiguous bf16 tensor of n * 2 pages")
    desc = make_desc(k_cache, k_cache.shape[1], 1)
    with torch.cuda.device(k_cache.device):
        _check(lib().pkv_export_pages(_ptr(k_cache), _ptr(v_cache), _ptr(pages), n, _ptr(out),
                                      ctypes.byref(desc), _stream(k_cache.device, stream)), "pkv_export_pages")
    return out


def import_pages(src, pages, k_cache, v_cache, stream=None):
    """Copy a buffer written by export_pages into the listed pool pages."""
    _need(pages, "pages", torch.int32, 1)
    n = pages.shape[0]
    if src.dtype != torch.bfloat16 or not src.is_contiguous() or src.numel() != n * 2 * k_cache[0].numel():
        raise ValueError("src must be a contiguous bf16 tensor of n * 2 pages")
    desc = make_desc(k_cache, k_cache.shape[1], 1)
    with torch.cuda.device(k_cache.device):
        _check(lib().pkv_import_pages(_ptr(src), _ptr(pages), n, _ptr(k_cache), _ptr(v_cache),
                                      ctypes.byref(desc), _stream(k_cache.device, stream)), "pkv_import_pages")


def get_last_error(device=None, stream=None):
    """Wait for the stream; read and clear the device status bits."""
    flags = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().pkv_get_last_error(_stream(dev, stream), ctypes.byref(flags)), "pkv_get_last_error")
    return flags.value


def launch_count():
    return int(lib().pkv_launch_count())


class PagePool:
    """Host-side page allocator with reference counts (see pkv_pool_* in pkv.h)."""

    def __init__(self, num_blocks):
        h = ctypes.c_void_p()
        _check(lib().pkv_pool_create(int(num_blocks), ctypes.byref(h)), "pkv_pool_create")
        self._h, self.num_blocks = h, int(num_blocks)

    @staticmethod
    def _arr(pages):
        pages = [int(x) for x in pages]
        return (ctypes.c_int32 * max(1, len(pages)))(*pages), len(pages)

    def alloc(self, n):
        buf = (ctypes.c_int32 * max(1, n))()
        _check(lib().pkv_pool_alloc(self._h, int(n), buf), "pkv_pool_alloc")
        return list(buf)[:n]

    def retain(self, pages):
        a, n = self._arr(pages)
        _check(lib().pkv_pool_retain(self._h, a, n), "pkv_pool_retain")

    def release(self, pages):
        a, n = self._arr(pages)
        _check(lib().pkv_pool_release(self._h, a, n), "pkv_pool_release")

    def refcount(self, page):
        c = ctypes.c_int32(0)
        _check(lib().pkv_pool_refcount(self._h, int(page), ctypes.byref(c)), "pkv_pool_refcount")
        return c.value

    def usage(self):
        u, t = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib().pkv_pool_usage(self._h, ctypes.byref(u), ctypes.byref(t)), "pkv_pool_usage")
        return u.value, t.value

    def make_writable(self, page, rows, k_cache, v_cache, stream=None):
        """Private copy of a shared page (copy-on-write); returns the page to write."""
        desc = make_desc(k_cache, k_cache.shape[1], 1)
        out = ctypes.c_int32(-1)
        with torch.cuda.device(k_cache.device):
            _check(lib().pkv_pool_make_writable(self._h, int(page), int(rows), _ptr(k_cache), _ptr(v_cache),
                                                ctypes.byref(desc), _stream(k_cache.device, stream),
                                                ctypes.byref(out)), "pkv_pool_make_writable")
        return out.value

    def close(self):
        if self._h:
            lib().pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Trace:
    """Per-kernel device time of the library's launches on this thread."""

    def __init__(self, capacity=4096):
        h = ctypes.c_void_p()
        _check(lib().pkv_trace_create(capacity, ctypes.byref(h)), "pkv_trace_create")
        self._h = h

    def __enter__(self):
        _check(lib().pkv_trace_attach(self._h), "pkv_trace_attach")
        return self

    def __exit__(self, *exc):
        lib().pkv_trace_detach()
        return False

    def read(self, kernel):
        ms, n = ctypes.c_double(0), ctypes.c_int64(0)
        kid = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
        _check(lib().pkv_trace_read(self._h, kid, ctypes.byref(ms), ctypes.byref(n)), "pkv_trace_read")
        return ms.value, n.value

    def reset(self):
        _check(lib().pkv_trace_reset(self._h), "pkv_trace_reset")

    def close(self):
        if self._h:
            lib().pkv_trace_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
