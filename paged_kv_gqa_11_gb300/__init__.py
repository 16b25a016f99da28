"""Paged GQA decode attention on GB300: Python binding of libpa.

A thin ctypes layer over the C ABI declared in ``include/pa.h``: it marshals
pointers, sizes and the current CUDA stream and returns status codes.  All the
work -- allocation bookkeeping, the append scatter, the split decode and its
merge -- runs inside libpa (host C++ and sm_103a CUDA kernels).  There is no
Python or CPU fallback: if libpa has not been built, every call raises.

Device buffers are torch tensors (torch owns the memory); the library never
allocates device memory.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import _build

__all__ = [
    "PA_F16", "PA_Q4_0", "PA_Q8_0", "PaError", "Pool", "load", "row_bytes", "pa_append_rows", "pa_append_rows_f16", "pa_copy_blocks", "pa_decode",
    "pa_decode_workspace_size", "pa_decode_plan", "pa_get_error", "pa_selftest_wait_timeout", "status_name",
    "library_path", "pa_decode_noalloc",
]

PA_F16, PA_Q4_0, PA_Q8_0 = 1, 2, 8
STATUS = ["PA_OK", "PA_ERR_INVALID", "PA_ERR_UNSUPPORTED", "PA_ERR_OOM", "PA_ERR_STALE", "PA_ERR_BOUNDS",
          "PA_ERR_TIMEOUT", "PA_ERR_CUDA"]
PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_OOM, PA_ERR_STALE, PA_ERR_BOUNDS, PA_ERR_TIMEOUT, PA_ERR_CUDA = range(8)

# Every entry point declared in include/pa.h.
EXPORTS = ["pa_pool_create", "pa_pool_destroy", "pa_pool_get_desc", "pa_row_bytes", "pa_pool_bytes",
           "pa_alloc_blocks", "pa_release", "pa_block_index", "pa_pool_free_count", "pa_share_blocks", "pa_block_refcount",
           "pa_cow_blocks", "pa_copy_blocks", "pa_append_rows", "pa_append_rows_f16",
           "pa_decode", "pa_decode_split", "pa_decode_merge", "pa_decode_workspace_size", "pa_decode_plan", "pa_get_error", "pa_status_string",
           "pa_selftest_wait_timeout", "pa_decode_noalloc"]


class PaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_name(status)}" if what else status_name(status))


def status_name(s: int) -> str:
    return STATUS[s] if 0 <= s < len(STATUS) else f"PA_STATUS_{s}"


class PoolDesc(C.Structure):
    _fields_ = [("n_blocks", C.c_uint32), ("page_size", C.c_uint32), ("n_kv_heads", C.c_uint32),
                ("head_dim", C.c_uint32), ("k_type", C.c_int32), ("v_type", C.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libpa.so; raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libpa is not built ({path} missing); run paged_kv_gqa_11_gb300._build.build()")
        L = C.CDLL(path)
        vp, u32, i32, sz = C.c_void_p, C.c_uint32, C.c_int32, C.c_size_t
        sig = {
            "pa_pool_create": (C.c_int, [C.POINTER(PoolDesc), C.POINTER(vp)]),
            "pa_pool_destroy": (None, [vp]),
            "pa_pool_get_desc": (C.c_int, [vp, C.POINTER(PoolDesc)]),
            "pa_row_bytes": (sz, [i32, u32]),
            "pa_pool_bytes": (sz, [vp, C.c_int]),
            "pa_alloc_blocks": (C.c_int, [vp, u32, vp]),
            "pa_release": (C.c_int, [vp, vp, u32]),
            "pa_block_index": (C.c_int, [vp, C.c_uint64, C.POINTER(i32)]),
            "pa_pool_free_count": (u32, [vp]),
            "pa_share_blocks": (C.c_int, [vp, vp, u32]),
            "pa_block_refcount": (C.c_int, [vp, C.c_uint64, C.POINTER(u32)]),
            "pa_cow_blocks": (C.c_int, [vp, vp, u32, vp, vp, vp, C.POINTER(u32)]),
            "pa_copy_blocks": (C.c_int, [vp, vp, vp, vp, vp, u32, vp, vp]),
            "pa_append_rows": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, u32, vp, u32, u32, vp, vp]),
            "pa_append_rows_f16": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, u32, vp, u32, u32, vp, vp]),
            "pa_decode": (C.c_int, [vp, vp, vp, vp, vp, u32, vp, vp, u32, u32, u32, C.c_float, vp, vp, vp, sz,
                                    vp, vp]),
            "pa_decode_workspace_size": (sz, [vp, u32, u32, C.c_int]),
            "pa_decode_plan": (C.c_int, [vp, vp, u32, u32, C.c_int, C.POINTER(u32), C.POINTER(u32),
                                         C.POINTER(u32), C.POINTER(u32)]),
            "pa_get_error": (C.c_int, [vp, vp]),
            "pa_status_string": (C.c_char_p, [C.c_int]),
            "pa_selftest_wait_timeout": (C.c_int, [u32, vp, vp]),
            "pa_decode_noalloc": (C.c_int, [vp, vp, vp, vp, vp, u32, vp, vp, u32, u32, u32, C.c_float, vp, vp,
                                            vp, vp]),
        }
        sig["pa_decode_split"] = sig["pa_decode_merge"] = sig["pa_decode"]
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return L


def row_bytes(t: int, head_dim: int = 256) -> int:
    return int(load().pa_row_bytes(t, head_dim))


def _ptr(x) -> int | None:
    """Device/host address of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str) -> None:
    if rc != PA_OK:
        raise PaError(rc, what)


class Pool:
    """Allocator state of one K/V pool (host metadata; see pa_pool_create)."""

    def __init__(self, n_blocks: int, page_size: int, n_kv_heads: int = 4, head_dim: int = 256,
                 k_type: int = PA_F16, v_type: int | None = None):
        L = load()
        self.desc = PoolDesc(n_blocks, page_size, n_kv_heads, head_dim, k_type,
                             k_type if v_type is None else v_type)
        h = C.c_void_p()
        _check(L.pa_pool_create(C.byref(self.desc), C.byref(h)), "pa_pool_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            load().pa_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def bytes(self, which: int) -> int:
        return int(load().pa_pool_bytes(self._h, which))

    def alloc(self, n: int) -> list[int]:
        buf = (C.c_uint64 * max(n, 1))()
        _check(load().pa_alloc_blocks(self._h, n, buf), "pa_alloc_blocks")
        return list(buf[:n])

    def alloc_status(self, n: int):
        buf = (C.c_uint64 * max(n, 1))()
        rc = load().pa_alloc_blocks(self._h, n, buf)
        return rc, (list(buf[:n]) if rc == PA_OK else [])

    def release(self, handles) -> int:
        arr = (C.c_uint64 * max(len(handles), 1))(*handles)
        return int(load().pa_release(self._h, arr, len(handles)))

    def block_index(self, handle: int):
        idx = C.c_int32(-1)
        rc = load().pa_block_index(self._h, handle, C.byref(idx))
        return rc, idx.value

    def free_count(self) -> int:
        return int(load().pa_pool_free_count(self._h))

    def share(self, handles) -> int:
        arr = (C.c_uint64 * max(len(handles), 1))(*handles)
        return int(load().pa_share_blocks(self._h, arr, len(handles)))

    def refcount(self, handle: int):
        n = C.c_uint32(0)
        rc = load().pa_block_refcount(self._h, handle, C.byref(n))
        return rc, n.value

    def cow(self, handles):
        """Returns (status, handles to write through, [(src index, dst index)] copies)."""
        k = max(len(handles), 1)
        arr = (C.c_uint64 * k)(*handles)
        out = (C.c_uint64 * k)()
        src, dst = (C.c_int32 * k)(), (C.c_int32 * k)()
        nc = C.c_uint32(0)
        rc = int(load().pa_cow_blocks(self._h, arr, len(handles), out, src, dst, C.byref(nc)))
        if rc != PA_OK:
            return rc, [], []
        return rc, list(out[:len(handles)]), [(src[i], dst[i]) for i in range(nc.value)]


def pa_append_rows(pool: Pool, k_pool, v_pool, k_rows, v_rows, row_seq, row_pos, n_rows: int, block_table,
                   table_stride: int, n_seq: int, err, stream=None) -> None:
    rc = load().pa_append_rows(pool.handle, _ptr(k_pool), _ptr(v_pool), _ptr(k_rows), _ptr(v_rows), _ptr(row_seq),
                               _ptr(row_pos), n_rows, _ptr(block_table), table_stride, n_seq, _ptr(err),
                               _stream(stream))
    _check(rc, "pa_append_rows")


def pa_append_rows_f16(pool: Pool, k_pool, v_pool, k_rows, v_rows, row_seq, row_pos, n_rows: int, block_table,
                       table_stride: int, n_seq: int, err, stream=None) -> None:
    """Rows as binary16 [n_rows][n_kv_heads][head_dim], quantised into the pool's formats."""
    rc = load().pa_append_rows_f16(pool.handle, _ptr(k_pool), _ptr(v_pool), _ptr(k_rows), _ptr(v_rows),
                                   _ptr(row_seq), _ptr(row_pos), n_rows, _ptr(block_table), table_stride, n_seq,
                                   _ptr(err), _stream(stream))
    _check(rc, "pa_append_rows_f16")


def pa_copy_blocks(pool: Pool, k_pool, v_pool, src, dst, n: int, err, stream=None) -> None:
    """Copy whole blocks src[i] -> dst[i] (device int32 arrays) in both pools."""
    rc = load().pa_copy_blocks(pool.handle, _ptr(k_pool), _ptr(v_pool), _ptr(src), _ptr(dst), n, _ptr(err),
                               _stream(stream))
    _check(rc, "pa_copy_blocks")


def pa_decode_workspace_size(pool: Pool, n_seq: int, n_qtok: int, device: int = 0) -> int:
    return int(load().pa_decode_workspace_size(pool.handle, n_seq, n_qtok, device))


def pa_decode_plan(pool: Pool, seq_lens_host, n_qtok: int, device: int = 0) -> dict:
    import numpy as np
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    a, b, c, d = C.c_uint32(), C.c_uint32(), C.c_uint32(), C.c_uint32()
    _check(load().pa_decode_plan(pool.handle, sl.ctypes.data, len(sl), n_qtok, device, C.byref(a), C.byref(b),
                                 C.byref(c), C.byref(d)), "pa_decode_plan")
    return {"ctas": a.value, "tiles": b.value, "tile_keys": c.value, "partials": d.value}


def pa_decode(pool: Pool, q, k_pool, v_pool, block_table, table_stride: int, seq_lens_dev, seq_lens_host,
              n_seq: int, n_qtok: int, n_q_heads: int, scale: float, out, lse, workspace, ws_bytes: int, err,
              stream=None, check: bool = True, passes: str = "all") -> int:
    """seq_lens_host: a host int32 buffer (numpy array or address) that stays
    alive for the call.  passes: "all" (pa_decode), "split" (pa_decode_split)
    or "merge" (pa_decode_merge)."""
    fn = {"all": "pa_decode", "split": "pa_decode_split", "merge": "pa_decode_merge"}[passes]
    rc = getattr(load(), fn)(pool.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), table_stride,
                          _ptr(seq_lens_dev), _ptr(seq_lens_host), n_seq, n_qtok, n_q_heads, C.c_float(scale),
                          _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(err), _stream(stream))
    if check:
        _check(rc, "pa_decode")
    return rc


def pa_get_error(err, stream=None) -> int:
    return int(load().pa_get_error(_ptr(err), _stream(stream)))


def pa_selftest_wait_timeout(timeout_us: int, err, stream=None) -> int:
    return int(load().pa_selftest_wait_timeout(timeout_us, _ptr(err), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def pa_decode_noalloc(pool: Pool, q, k_pool, v_pool, block_table, table_stride: int, seq_lens_dev, seq_lens_host,
                      n_seq: int, n_qtok: int, n_q_heads: int, scale: float, out, lse, err, stream=None) -> int:
    """pa_decode with the library's fixed scratch instead of a caller workspace
    (for callers that cannot allocate device memory); returns the status."""
    return int(load().pa_decode_noalloc(pool.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                        table_stride, _ptr(seq_lens_dev), _ptr(seq_lens_host), n_seq, n_qtok,
                                        n_q_heads, C.c_float(scale), _ptr(out), _ptr(lse), _ptr(err),
                                        _stream(stream)))
