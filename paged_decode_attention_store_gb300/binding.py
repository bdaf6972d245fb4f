"""Thin Python binding of libpagedkv (argument marshalling only).

Same names as the C ABI in ``include/pagedkv.h``. Device arguments are torch
CUDA tensors (PyTorch supplies device memory and streams); every step of the
path runs in the library's kernels. A missing library or a non-zero status
raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

KVP_OK = 0
KVP_ERR_INVALID_ARG = -1
KVP_ERR_CUDA = -2
KVP_ERR_OUT_OF_PAGES = -3
KVP_ERR_BAD_INDEX = -4
KVP_ERR_TIMEOUT = -5

KVP_F32, KVP_BF16 = 0, 1
KVP_BLOCK_TABLE, KVP_RAW_LOCATIONS = 0, 1

_ERR_NAMES = {
    KVP_ERR_INVALID_ARG: "KVP_ERR_INVALID_ARG",
    KVP_ERR_CUDA: "KVP_ERR_CUDA",
    KVP_ERR_OUT_OF_PAGES: "KVP_ERR_OUT_OF_PAGES",
    KVP_ERR_BAD_INDEX: "KVP_ERR_BAD_INDEX",
    KVP_ERR_TIMEOUT: "KVP_ERR_TIMEOUT",
}

# Every symbol the header declares, with its C signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)
_szp = ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "kv_pool_create": [_i, _i, _i, _i, _i, _i, _vp, _vp, ctypes.POINTER(_vp)],
    "kv_pool_destroy": [_vp],
    "store_cache": [_vp, _i, _vp, _vp, _vp, _i, _vp],
    "page_table_write": [_vp, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _vp],
    "copy_pages": [_vp, _vp, _vp, _i, _vp],
    "paged_decode_attention_workspace_size": [_vp, _i, _i, _szp],
    "paged_decode_attention": [_vp, _i, _vp, _i, _i, _vp, _i, _i, _i, _vp, _vp, _i, _i, _f, _vp, _vp, _sz, _vp],
    "paged_verify_attention_workspace_size": [_vp, _i, _i, _i, _szp],
    "paged_verify_attention": [_vp, _i, _vp, _i, _i, _i, _vp, _i, _i, _i, _vp, _vp, _i, _i, _f, _vp, _vp, _sz, _vp],
    "paged_prefill_attention": [_vp, _i, _vp, _i, _i, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _i, _i, _f, _vp, _vp],
    "paged_decode_attention_noalloc": [_vp, _i, _vp, _i, _i, _vp, _i, _i, _i, _vp, _vp, _i, _i, _f, _vp, _vp],
    "store_cache_and_attention": [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i,
                                  _i, _i, _f, _vp, _vp, _sz, _vp],
    "gather_indices": [_vp, _vp, _i, _i, _i, _vp, _vp, _i, _i, _i, _vp, _i, _vp],
    "kvp_sync_error": [_vp, _vp, _ip],
    "kvp_selftest_wait": [ctypes.c_longlong, _i, _vp, _vp],
    "kvp_pool_set_timing_events": [_vp, _vp, _vp],
    "kvp_host_create": [_i, _i, _i, _vp, ctypes.POINTER(_vp)],
    "kvp_host_destroy": [_vp],
    "kvp_host_new": [_vp, _i],
    "kvp_host_fork": [_vp, _i, _i, _vp, _vp, _vp, _i, _ip],
    "kvp_host_release": [_vp, _i],
    "kvp_host_append": [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _ip, _vp, _vp, _ip],
    "kvp_host_trim": [_vp, _i, _i, _vp, _vp, _vp, _i, _ip],
    "kvp_host_trim_sinks": [_vp, _i, _i, _i, _vp, _vp, _vp, _i, _ip],
    "kvp_host_rewind": [_vp, _i, _i, _vp, _vp, _vp, _i, _ip],
    "kvp_host_used": [_vp, _ip],
    "kvp_host_length": [_vp, _i, _ip, _ip],
    "kvp_host_block_row": [_vp, _i, _vp, _i, _ip],
    "kvp_host_refcounts": [_vp, _vp, _i],
    "kvp_host_free_list": [_vp, _vp, _i, _ip],
    "kvp_dev_pages_bytes": [_i, _i, _szp],
    "kvp_dev_pages_create": [_i, _i, _i, _vp, _sz, _vp, _i, _i, _i, ctypes.POINTER(_vp)],
    "kvp_dev_pages_destroy": [_vp],
    "kvp_dev_pages_init": [_vp, _vp, _vp],
    "kvp_dev_new": [_vp, _vp, _i, _vp],
    "kvp_dev_append": [_vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp],
    "kvp_dev_trim": [_vp, _vp, _vp, _i, _i, _i, _vp],
    "kvp_dev_release": [_vp, _vp, _i, _vp],
    "kvp_dev_sync_error": [_vp, _vp, _ip],
    "kvp_dev_fork": [_vp, _vp, _vp, _i, _vp],
    "kvp_dev_rewind": [_vp, _vp, _vp, _i, _vp],
    "kvp_verify_step_device_io": [_vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp],
    "copy_pages_device_count": [_vp, _vp, _vp, _vp, _i, _vp],
    "kvp_decode_step_device": [_vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp,
                               _vp, _i, _vp, _sz, _vp],
    "kvp_decode_step_device_io": [_vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _i, _vp, _sz, _vp],
    "kvp_decode_step": [_vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                        _i, _vp, _sz, _vp, _vp],
}


class StepInfo(ctypes.Structure):
    _fields_ = [("n_table_writes", ctypes.c_int), ("n_copies", ctypes.c_int), ("n_trim_writes", ctypes.c_int),
                ("meta_ints", ctypes.c_int)]

_lib = None


class KvpError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {_ERR_NAMES.get(code, code)}")
        self.code = code


class OutOfPages(KvpError):
    pass


def lib():
    """Load libpagedkv.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(code, what):
    if code == KVP_ERR_OUT_OF_PAGES:
        raise OutOfPages(code, what)
    if code != KVP_OK:
        raise KvpError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype=None, name="tensor"):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_TORCH_DTYPE = {KVP_F32: torch.float32, KVP_BF16: torch.bfloat16}


class Pool:
    """A kvp_pool over a caller-owned KV buffer (kept alive here)."""

    def __init__(self, kv_buffer, page_size, dtype, error_word=None):
        _dev(kv_buffer, name="kv_buffer")
        if kv_buffer.dim() != 6 or kv_buffer.shape[0] != 2 or kv_buffer.shape[3] != page_size:
            raise ValueError("kv_buffer must be (2, layers, num_pages, page_size, kv_heads, head_dim)")
        if kv_buffer.dtype != _TORCH_DTYPE[dtype]:
            raise TypeError("kv_buffer dtype does not match")
        _, self.num_layers, self.num_pages, self.page_size, self.kv_heads, self.head_dim = kv_buffer.shape
        self.dtype = dtype
        self.kv_buffer = kv_buffer
        self.error_word = (torch.zeros(1, dtype=torch.int32, device=kv_buffer.device)
                           if error_word is None else _dev(error_word, torch.int32, "error_word"))
        h = ctypes.c_void_p()
        _check(lib().kv_pool_create(self.num_pages, page_size, self.kv_heads, self.head_dim, dtype,
                                    self.num_layers, _ptr(kv_buffer), _ptr(self.error_word), ctypes.byref(h)),
               "kv_pool_create")
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.kv_pool_destroy(h)
            self.handle = None


def kv_pool_create(num_pages, page_size, kv_heads, head_dim, dtype, num_layers, kv_buffer=None, device="cuda"):
    """Describe (allocating with torch when ``kv_buffer`` is None) a KV buffer."""
    if kv_buffer is None:
        kv_buffer = torch.empty((2, num_layers, num_pages, page_size, kv_heads, head_dim),
                                dtype=_TORCH_DTYPE[dtype], device=device)
    return Pool(kv_buffer, page_size, dtype)


def store_cache(pool, layer, k, v, out_loc, stream=None):
    _dev(k, _TORCH_DTYPE[pool.dtype], "k")
    _dev(v, _TORCH_DTYPE[pool.dtype], "v")
    _dev(out_loc, torch.int32, "out_loc")
    n = out_loc.numel()
    if k.numel() != n * pool.kv_heads * pool.head_dim or v.numel() != k.numel():
        raise ValueError("k/v must be [n, kv_heads, head_dim]")
    _check(lib().store_cache(pool.handle, layer, _ptr(k), _ptr(v), _ptr(out_loc), n, _stream(stream)), "store_cache")


def page_table_write(table, rows, cols, vals, expand=1, error_word=None, stream=None):
    _dev(table, torch.int32, "table")
    for t, nm in ((rows, "rows"), (cols, "cols"), (vals, "vals")):
        _dev(t, torch.int32, nm)
    n = rows.numel()
    if cols.numel() != n or vals.numel() != n:
        raise ValueError("rows, cols and vals must have the same length")
    _check(lib().page_table_write(_ptr(table), table.shape[0], table.shape[1], _ptr(rows), _ptr(cols), _ptr(vals),
                                  n, expand, _ptr(error_word), _stream(stream)), "page_table_write")


class DevicePages:
    """Device-side page allocation over a caller's device table (see
    include/pagedkv.h, kvp_dev_*). The state buffer is allocated here with
    torch and kept alive; every call is asynchronous on the current stream."""

    def __init__(self, num_pages, page_size, max_requests, table, table_mode, free_stack=None, device="cuda"):
        _dev(table, torch.int32, "table")
        n = ctypes.c_size_t()
        _check(lib().kvp_dev_pages_bytes(num_pages, max_requests, ctypes.byref(n)), "kvp_dev_pages_bytes")
        self.state = torch.zeros(n.value, dtype=torch.uint8, device=device)
        self.table = table
        self.num_pages, self.page_size, self.max_requests = num_pages, page_size, max_requests
        h = ctypes.c_void_p()
        _check(lib().kvp_dev_pages_create(num_pages, page_size, max_requests, _ptr(self.state), n.value, _ptr(table),
                                          table.shape[0], table.shape[1], table_mode, ctypes.byref(h)),
               "kvp_dev_pages_create")
        self.handle = h
        fs = None
        if free_stack is not None:
            fs = torch.as_tensor(list(free_stack), dtype=torch.int32).to(device)
            if fs.numel() != num_pages:
                raise ValueError("free_stack must hold num_pages entries")
        self._free_stack = fs
        _check(lib().kvp_dev_pages_init(h, _ptr(fs), _stream(None)), "kvp_dev_pages_init")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.kvp_dev_pages_destroy(h)
            self.handle = None

    def new(self, rids, stream=None):
        _dev(rids, torch.int32, "rids")
        _check(lib().kvp_dev_new(self.handle, _ptr(rids), rids.numel(), _stream(stream)), "kvp_dev_new")

    def append(self, rids, out_loc, cow_src, cow_dst, n_cow, counts=None, lens_out=None, stream=None):
        for t, nm in ((rids, "rids"), (out_loc, "out_loc"), (cow_src, "cow_src"), (cow_dst, "cow_dst"),
                      (n_cow, "n_cow")):
            _dev(t, torch.int32, nm)
        if counts is not None:
            _dev(counts, torch.int32, "counts")
        n = rids.numel()
        if cow_src.numel() < n or cow_dst.numel() < n:
            raise ValueError("cow_src/cow_dst need room for one pair per request")
        if lens_out is not None:
            _dev(lens_out, torch.int32, "lens_out")
        _check(lib().kvp_dev_append(self.handle, _ptr(rids), _ptr(counts), n, _ptr(out_loc), out_loc.numel(),
                                    _ptr(cow_src), _ptr(cow_dst), _ptr(n_cow), _ptr(lens_out), _stream(stream)),
               "kvp_dev_append")

    def trim(self, rids, keep_from=None, sinks=0, window=0, stream=None):
        """Release what the next step cannot read: below keep_from[i] (device
        int32), or, without keep_from, below each request's L + 1 - (window - sinks)."""
        _dev(rids, torch.int32, "rids")
        if keep_from is not None:
            _dev(keep_from, torch.int32, "keep_from")
        _check(lib().kvp_dev_trim(self.handle, _ptr(rids), _ptr(keep_from), rids.numel(), int(window), int(sinks),
                                  _stream(stream)), "kvp_dev_trim")

    def release(self, rids, stream=None):
        _dev(rids, torch.int32, "rids")
        _check(lib().kvp_dev_release(self.handle, _ptr(rids), rids.numel(), _stream(stream)), "kvp_dev_release")

    def fork(self, src, dst, stream=None):
        _dev(src, torch.int32, "src")
        _dev(dst, torch.int32, "dst")
        if src.numel() != dst.numel():
            raise ValueError("src and dst must have the same length")
        _check(lib().kvp_dev_fork(self.handle, _ptr(src), _ptr(dst), src.numel(), _stream(stream)), "kvp_dev_fork")

    def rewind(self, rids, n_back, stream=None):
        """Drop the newest n_back[i] rows of request rids[i] (both device int32)."""
        _dev(rids, torch.int32, "rids")
        _dev(n_back, torch.int32, "n_back")
        if rids.numel() != n_back.numel():
            raise ValueError("rids and n_back must have the same length")
        _check(lib().kvp_dev_rewind(self.handle, _ptr(rids), _ptr(n_back), rids.numel(), _stream(stream)),
               "kvp_dev_rewind")

    def sync_error(self, stream=None):
        e = ctypes.c_int()
        _check(lib().kvp_dev_sync_error(self.handle, _stream(stream), ctypes.byref(e)), "kvp_dev_sync_error")
        return e.value

    def snapshot(self):
        """(free list, reference counts, lengths, released pages, sink pages) read back to the host."""
        P, R = self.num_pages, self.max_requests
        a16 = lambda x: (x + 15) // 16 * 16  # noqa: E731
        st = self.state.cpu()
        hdr = st[:16].view(torch.int32).tolist()
        off = 16
        stack = st[off:off + 4 * P].view(torch.int32).tolist()
        off += a16(4 * P)
        ref = st[off:off + 4 * P].view(torch.int32).tolist()
        off += a16(4 * P)
        arr = []
        for _ in range(3):
            arr.append(st[off:off + 4 * R].view(torch.int32).tolist())
            off += a16(4 * R)
        return stack[:hdr[0]], ref, arr[0], arr[1], arr[2]


def copy_pages_device_count(pool, src, dst, n_dev, stream=None):
    _dev(src, torch.int32, "src")
    _dev(dst, torch.int32, "dst")
    _dev(n_dev, torch.int32, "n_dev")
    _check(lib().copy_pages_device_count(pool.handle, _ptr(src), _ptr(dst), _ptr(n_dev), src.numel(),
                                         _stream(stream)), "copy_pages_device_count")


def copy_pages(pool, src, dst, stream=None):
    _dev(src, torch.int32, "src")
    _dev(dst, torch.int32, "dst")
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same length")
    _check(lib().copy_pages(pool.handle, _ptr(src), _ptr(dst), src.numel(), _stream(stream)), "copy_pages")


def paged_decode_attention_workspace_size(pool, batch, num_q_heads):
    n = ctypes.c_size_t()
    _check(lib().paged_decode_attention_workspace_size(pool.handle, batch, num_q_heads, ctypes.byref(n)),
           "paged_decode_attention_workspace_size")
    return n.value


def alloc_workspace(pool, batch, num_q_heads, device="cuda"):
    nbytes = paged_decode_attention_workspace_size(pool, batch, num_q_heads)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def paged_decode_attention(pool, layer, q, table, table_mode, context_lens, window, scale, out, workspace,
                           table_rows=None, stream=None, sinks=0):
    dt = _TORCH_DTYPE[pool.dtype]
    _dev(q, dt, "q")
    _dev(out, dt, "out")
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    if table_rows is not None:
        _dev(table_rows, torch.int32, "table_rows")
    B, Hq = q.shape[0], q.shape[1]
    if out.shape != q.shape or context_lens.numel() != B:
        raise ValueError("q/out must be [B, Hq, D] and context_lens [B]")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(lib().paged_decode_attention(pool.handle, layer, _ptr(q), B, Hq, _ptr(table), table.shape[0],
                                        table.shape[1], table_mode, _ptr(table_rows), _ptr(context_lens),
                                        int(window or 0), int(sinks), float(scale), _ptr(out), ws_ptr, ws_bytes,
                                        _stream(stream)), "paged_decode_attention")


def paged_verify_attention_workspace_size(pool, batch, num_q_tokens, num_q_heads):
    n = ctypes.c_size_t()
    _check(lib().paged_verify_attention_workspace_size(pool.handle, batch, num_q_tokens, num_q_heads,
                                                       ctypes.byref(n)), "paged_verify_attention_workspace_size")
    return n.value


def alloc_verify_workspace(pool, batch, num_q_tokens, num_q_heads, device="cuda"):
    nbytes = paged_verify_attention_workspace_size(pool, batch, num_q_tokens, num_q_heads)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def paged_verify_attention(pool, layer, q, table, table_mode, context_lens, window, scale, out, workspace,
                           table_rows=None, stream=None, sinks=0):
    """Multi-token verify: q/out [B, M, Hq, D]; query j of request b sits at
    position context_lens[b] - M + j and attends causally (see
    include/pagedkv.h)."""
    dt = _TORCH_DTYPE[pool.dtype]
    _dev(q, dt, "q")
    _dev(out, dt, "out")
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    if table_rows is not None:
        _dev(table_rows, torch.int32, "table_rows")
    if q.dim() != 4 or out.shape != q.shape or context_lens.numel() != q.shape[0]:
        raise ValueError("q/out must be [B, M, Hq, D] and context_lens [B]")
    B, M, Hq = q.shape[0], q.shape[1], q.shape[2]
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(lib().paged_verify_attention(pool.handle, layer, _ptr(q), B, M, Hq, _ptr(table), table.shape[0],
                                        table.shape[1], table_mode, _ptr(table_rows), _ptr(context_lens),
                                        int(window or 0), int(sinks), float(scale), _ptr(out), ws_ptr, ws_bytes,
                                        _stream(stream)), "paged_verify_attention")


def paged_prefill_attention(pool, layer, q, table, table_mode, context_lens, window, scale, out, q_lens=None,
                            table_rows=None, stream=None, sinks=0):
    """Chunked prefill: q/out [B, C, Hq, D]; query j of request b sits at
    position context_lens[b] - q_lens[b] + j (q_lens NULL: C) and attends
    causally (see include/pagedkv.h). Rows j >= q_lens[b] are not written."""
    dt = _TORCH_DTYPE[pool.dtype]
    _dev(q, dt, "q")
    _dev(out, dt, "out")
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    for t, nm in ((q_lens, "q_lens"), (table_rows, "table_rows")):
        if t is not None:
            _dev(t, torch.int32, nm)
    if q.dim() != 4 or out.shape != q.shape or context_lens.numel() != q.shape[0]:
        raise ValueError("q/out must be [B, C, Hq, D] and context_lens [B]")
    B, C, Hq = q.shape[0], q.shape[1], q.shape[2]
    _check(lib().paged_prefill_attention(pool.handle, layer, _ptr(q), B, C, Hq, _ptr(q_lens), _ptr(table),
                                         table.shape[0], table.shape[1], table_mode, _ptr(table_rows),
                                         _ptr(context_lens), int(window or 0), int(sinks), float(scale), _ptr(out),
                                         _stream(stream)), "paged_prefill_attention")


def store_cache_and_attention(pool, layer, q, k, v, out_loc, table, table_mode, context_lens, window, scale, out,
                              workspace, table_rows=None, table_writes=None, stream=None, sinks=0):
    """store_cache + paged_decode_attention of one layer in one launch, with
    the step's new-page table writes (rows, cols, vals device int32 tensors)
    applied in the same launch. out_loc[b] must be the slot of request b's
    newest position; see include/pagedkv.h for what the table writes may be."""
    dt = _TORCH_DTYPE[pool.dtype]
    for name, x in (("q", q), ("k", k), ("v", v), ("out", out)):
        _dev(x, dt, name)
    _dev(out_loc, torch.int32, "out_loc")
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    if table_rows is not None:
        _dev(table_rows, torch.int32, "table_rows")
    B, Hq = q.shape[0], q.shape[1]
    if out.shape != q.shape or context_lens.numel() != B or out_loc.numel() != B or k.shape[0] != B:
        raise ValueError("q/out [B, Hq, D], k/v [B, Hkv, D], out_loc and context_lens [B]")
    if table_writes is None:
        tw = (None, None, None, 0)
    else:
        r, c, vals = table_writes
        for name, x in (("rows", r), ("cols", c), ("vals", vals)):
            _dev(x, torch.int32, name)
        tw = (_ptr(r), _ptr(c), _ptr(vals), r.numel())
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(lib().store_cache_and_attention(pool.handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(out_loc), B, Hq,
                                           _ptr(table), table.shape[0], table.shape[1], table_mode,
                                           _ptr(table_rows), _ptr(context_lens), *tw, int(window or 0), int(sinks),
                                           float(scale), _ptr(out), ws_ptr, ws_bytes, _stream(stream)),
           "store_cache_and_attention")


def paged_decode_attention_noalloc(pool, layer, q, table, table_mode, context_lens, window, scale, out,
                                   table_rows=None, stream=None, sinks=0):
    """paged_decode_attention without a workspace argument, for callers that
    cannot allocate: the library uses a fixed scratch array of its own (see
    include/pagedkv.h). Overlapping calls on one device must be serialised."""
    dt = _TORCH_DTYPE[pool.dtype]
    _dev(q, dt, "q")
    _dev(out, dt, "out")
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    if table_rows is not None:
        _dev(table_rows, torch.int32, "table_rows")
    B, Hq = q.shape[0], q.shape[1]
    if out.shape != q.shape or context_lens.numel() != B:
        raise ValueError("q/out must be [B, Hq, D] and context_lens [B]")
    _check(lib().paged_decode_attention_noalloc(pool.handle, layer, _ptr(q), B, Hq, _ptr(table), table.shape[0],
                                                table.shape[1], table_mode, _ptr(table_rows), _ptr(context_lens),
                                                int(window or 0), int(sinks), float(scale), _ptr(out),
                                                _stream(stream)),
           "paged_decode_attention_noalloc")


def gather_indices(pool, table, table_mode, context_lens, window, slots_out, table_rows=None, stream=None, sinks=0):
    _dev(table, torch.int32, "table")
    _dev(context_lens, torch.int32, "context_lens")
    _dev(slots_out, torch.int32, "slots_out")
    B = context_lens.numel()
    _check(lib().gather_indices(pool.handle, _ptr(table), table.shape[0], table.shape[1], table_mode,
                                _ptr(table_rows), _ptr(context_lens), B, int(window or 0), int(sinks), _ptr(slots_out),
                                slots_out.shape[1], _stream(stream)), "gather_indices")


def kvp_pool_set_timing_events(pool, before=None, after=None):
    """Record ``before``/``after`` (torch.cuda.Event) around the next attention kernel."""
    b = None if before is None else ctypes.c_void_p(before.cuda_event)
    a = None if after is None else ctypes.c_void_p(after.cuda_event)
    _check(lib().kvp_pool_set_timing_events(pool.handle, b, a), "kvp_pool_set_timing_events")


def kvp_sync_error(pool, stream=None):
    e = ctypes.c_int()
    _check(lib().kvp_sync_error(pool.handle, _stream(stream), ctypes.byref(e)), "kvp_sync_error")
    return e.value


def kvp_selftest_wait(limit_ns, arrive, err, stream=None):
    """One bounded mbarrier wait on the device (kvp_selftest_wait): ``err`` is
    a device int32 tensor that receives KVP_ERR_TIMEOUT when nothing arrives."""
    _check(lib().kvp_selftest_wait(int(limit_ns), int(arrive), _ptr(err), _stream(stream)), "kvp_selftest_wait")


# ---------------------------------------------------------------------------
# Host bookkeeping (pure C++, usable without a GPU).
# ---------------------------------------------------------------------------
def _i32(n):
    return (ctypes.c_int32 * max(1, n))()


class HostPageTable:
    """kvp_host_*: refcounted LIFO free list, block tables with -1 holes,
    fork, lazy copy-on-write, window trim; emits device table writes."""

    def __init__(self, num_pages, page_size, max_requests, free_stack=None):
        self.num_pages, self.page_size, self.max_requests = num_pages, page_size, max_requests
        h = ctypes.c_void_p()
        fs = None
        if free_stack is not None:
            fs = (ctypes.c_int32 * num_pages)(*[int(x) for x in free_stack])
        _check(lib().kvp_host_create(num_pages, page_size, max_requests, fs, ctypes.byref(h)), "kvp_host_create")
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.kvp_host_destroy(h)
            self.handle = None

    def new(self, rid):
        _check(lib().kvp_host_new(self.handle, rid), "kvp_host_new")

    def fork(self, src, dst):
        """Share every page of ``src`` with ``dst``; returns the table writes for dst's row."""
        cap = self.length(src)[0] // self.page_size + 2
        tr, tc, tv = _i32(cap), _i32(cap), _i32(cap)
        n = ctypes.c_int()
        _check(lib().kvp_host_fork(self.handle, src, dst, tr, tc, tv, cap, ctypes.byref(n)), "kvp_host_fork")
        return list(zip(tr[:n.value], tc[:n.value], tv[:n.value]))

    def release(self, rid):
        _check(lib().kvp_host_release(self.handle, rid), "kvp_host_release")

    def append(self, rids):
        """One token for each entry of ``rids`` -> (slots, table writes, cow pairs) as Python lists."""
        rids = [int(r) for r in rids]
        n = len(rids)
        r = (ctypes.c_int32 * max(1, n))(*rids)
        slots, tr, tc, tv, cs, cd = _i32(n), _i32(n), _i32(n), _i32(n), _i32(n), _i32(n)
        ntw, ncow = ctypes.c_int(), ctypes.c_int()
        _check(lib().kvp_host_append(self.handle, r, n, slots, tr, tc, tv, n, ctypes.byref(ntw), cs, cd,
                                     ctypes.byref(ncow)), "kvp_host_append")
        writes = list(zip(tr[:ntw.value], tc[:ntw.value], tv[:ntw.value]))
        cows = list(zip(cs[:ncow.value], cd[:ncow.value]))
        return list(slots[:n]), writes, cows

    def append_into(self, rids, slots, tw, cow):
        """Fast form of :meth:`append` over numpy buffers.

        ``rids`` int32[n]; outputs go to ``slots`` int32[n], ``tw`` int32[3, n]
        (rows, cols, vals) and ``cow`` int32[2, n] (src, dst). Returns the
        numbers of table writes and copy-on-write pairs."""
        n = int(rids.shape[0])
        ntw, ncow = ctypes.c_int(), ctypes.c_int()
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
        _check(lib().kvp_host_append(self.handle, p(rids), n, p(slots), p(tw[0]), p(tw[1]), p(tw[2]), n,
                                     ctypes.byref(ntw), p(cow[0]), p(cow[1]), ctypes.byref(ncow)), "kvp_host_append")
        return ntw.value, ncow.value

    def trim_into(self, rid, keep_from, tw, cap, sinks=0):
        """Fast form of :meth:`trim`: writes go to ``tw`` int32[3, cap]; returns their number."""
        n = ctypes.c_int()
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
        _check(lib().kvp_host_trim_sinks(self.handle, rid, int(keep_from), int(sinks), p(tw[0]), p(tw[1]),
                                         p(tw[2]), cap, ctypes.byref(n)), "kvp_host_trim_sinks")
        return n.value

    def trim(self, rid, keep_from, sinks=0):
        """Release the pages no later step reads: below keep_from, except the
        first ceil(sinks / P) pages. Returns the (rid, page, -1) table writes."""
        cap = max(1, self.length(rid)[0] // self.page_size + 1)
        tr, tc, tv = _i32(cap), _i32(cap), _i32(cap)
        n = ctypes.c_int()
        if sinks:
            _check(lib().kvp_host_trim_sinks(self.handle, rid, int(keep_from), int(sinks), tr, tc, tv, cap,
                                             ctypes.byref(n)), "kvp_host_trim_sinks")
        else:
            _check(lib().kvp_host_trim(self.handle, rid, int(keep_from), tr, tc, tv, cap, ctypes.byref(n)),
                   "kvp_host_trim")
        return list(zip(tr[:n.value], tc[:n.value], tv[:n.value]))

    def rewind(self, rid, n):
        """Drop the newest n tokens; returns the (rid, page, -1) table writes
        of the pages let go (tail first)."""
        cap = max(1, self.length(rid)[0] // self.page_size + 1)
        tr, tc, tv = _i32(cap), _i32(cap), _i32(cap)
        k = ctypes.c_int()
        _check(lib().kvp_host_rewind(self.handle, rid, int(n), tr, tc, tv, cap, ctypes.byref(k)), "kvp_host_rewind")
        return list(zip(tr[:k.value], tc[:k.value], tv[:k.value]))

    def used(self):
        u = ctypes.c_int()
        _check(lib().kvp_host_used(self.handle, ctypes.byref(u)), "kvp_host_used")
        return u.value

    def length(self, rid):
        L, d = ctypes.c_int(), ctypes.c_int()
        _check(lib().kvp_host_length(self.handle, rid, ctypes.byref(L), ctypes.byref(d)), "kvp_host_length")
        return L.value, d.value

    def block_row(self, rid):
        L, _ = self.length(rid)
        cap = L // self.page_size + 2
        out = _i32(cap)
        n = ctypes.c_int()
        _check(lib().kvp_host_block_row(self.handle, rid, out, cap, ctypes.byref(n)), "kvp_host_block_row")
        return list(out[:n.value])

    def refcounts(self):
        out = _i32(self.num_pages)
        _check(lib().kvp_host_refcounts(self.handle, out, self.num_pages), "kvp_host_refcounts")
        return list(out[:self.num_pages])

    def free_list(self):
        out = _i32(self.num_pages)
        n = ctypes.c_int()
        _check(lib().kvp_host_free_list(self.handle, out, self.num_pages, ctypes.byref(n)), "kvp_host_free_list")
        return list(out[:n.value])
