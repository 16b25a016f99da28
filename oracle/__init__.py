"""Float64 CPU oracle for paged GQA decode attention -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library (``paged_kv_gqa_11_gb300``) never does, and
the oracle never imports the library: they share no code.  Inputs come from
the ``workloads`` generators, which hold no decode arithmetic.

The arithmetic lives in plain C (``pa_oracle.c``, float64, scalar loops);
this module compiles it with gcc and wraps it with ctypes.  The allocator
model is plain Python (``allocator_model.py``).

Pins (what keeps the oracle honest, all in the CPU test suite):
  * fp16 decode against numpy's independent binary16 implementation, every
    bit pattern;
  * dequantisation against hand-built blocks with known values, and the Q4_0
    block size against the capacity table of lucebox PR #555;
  * attention against closed forms (one key, identical keys, zero query,
    a dominant key, per-KV-head constants for the GQA mapping, causal
    visibility) and against a dense numpy/scipy brute force on tiny inputs;
  * invariants: shuffled placement and any page size give identical output;
    split-merge equals the unsplit softmax.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from contextlib import contextmanager

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liborc.so")
_lock = threading.Lock()
_lib = None

F16, Q4_0, Q8_0 = 1, 2, 8
ROLE_K, ROLE_V = 0, 1
GROUP = 16  # slots per row group of the pool layout


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math", "-ffp-contract=off",
            _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(src_text: str, tag: str) -> str:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    src = os.path.join(_OUT_DIR, f"variant_{tag}.c")
    out = os.path.join(_OUT_DIR, f"liborc_{tag}.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", src, "-o", out, "-lm"],
                   check=True, capture_output=True)
    return out


def source() -> str:
    with open(_SRC) as f:
        return f.read()


class _Cache(C.Structure):
    _fields_ = [("n_seq", C.c_int), ("n_qtok", C.c_int), ("hq", C.c_int), ("hkv", C.c_int),
                ("d", C.c_int), ("page_size", C.c_int), ("n_blocks", C.c_long),
                ("k_type", C.c_int), ("v_type", C.c_int),
                ("table", C.c_void_p), ("table_stride", C.c_long), ("seq_lens", C.c_void_p),
                ("k_pool", C.c_void_p), ("v_pool", C.c_void_p)]


def _load(path):
    L = C.CDLL(path)
    L.orc_half_to_double.restype = C.c_double
    L.orc_half_to_double.argtypes = [C.c_uint16]
    L.orc_row_bytes.restype = C.c_long
    L.orc_row_bytes.argtypes = [C.c_int, C.c_int]
    L.orc_dequant_row.restype = C.c_int
    L.orc_dequant_row.argtypes = [C.c_int, C.c_void_p, C.c_int, C.c_void_p]
    L.orc_attend_range.restype = C.c_int
    L.orc_attend_range.argtypes = [C.POINTER(_Cache), C.c_void_p, C.c_double, C.c_int, C.c_int,
                                   C.c_int, C.c_long, C.c_long, C.c_void_p,
                                   C.POINTER(C.c_double), C.POINTER(C.c_double)]
    L.orc_merge.restype = None
    L.orc_merge.argtypes = [C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                            C.POINTER(C.c_double)]
    L.orc_decode.restype = C.c_int
    L.orc_decode.argtypes = [C.POINTER(_Cache), C.c_void_p, C.c_double, C.c_void_p, C.c_void_p,
                             C.c_void_p, C.c_int]
    L.orc_scatter.restype = C.c_int
    L.orc_scatter.argtypes = [C.c_void_p, C.c_long, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                              C.c_void_p, C.c_void_p, C.c_void_p, C.c_long, C.c_void_p, C.c_long, C.c_int]
    L.orc_float_to_half.restype = C.c_uint16
    L.orc_float_to_half.argtypes = [C.c_float]
    L.orc_quantize_block.restype = C.c_int
    L.orc_quantize_block.argtypes = [C.c_int, C.c_void_p, C.c_void_p]
    L.orc_group_offset.restype = C.c_long
    L.orc_group_offset.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_long]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


@contextmanager
def using(path: str):
    """Temporarily route every oracle call through the library at `path`."""
    global _lib
    prev = lib()
    with _lock:
        _lib = _load(path)
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def half_to_double(bits: np.ndarray) -> np.ndarray:
    L = lib()
    bits = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([L.orc_half_to_double(int(b)) for b in bits], dtype=np.float64)


def row_bytes(t: int, d: int = 256) -> int:
    return int(lib().orc_row_bytes(t, d))


def dequant_rows(rows: np.ndarray, t: int, d: int = 256) -> np.ndarray:
    """uint8 [..., row_bytes] -> float64 [..., d]."""
    L = lib()
    rb = row_bytes(t, d)
    r = np.ascontiguousarray(rows, dtype=np.uint8).reshape(-1, rb)
    out = np.empty((r.shape[0], d), np.float64)
    for i in range(r.shape[0]):
        rc = L.orc_dequant_row(t, _ptr(r[i]), d, _ptr(out[i]))
        if rc:
            raise ValueError(f"orc_dequant_row rc={rc}")
    return out.reshape(*rows.shape[:-1], d)


def float_to_half(x) -> np.ndarray:
    """float32 values -> binary16 bit patterns (uint16), round to nearest even."""
    L = lib()
    xs = np.asarray(x, dtype=np.float32).ravel()
    return np.array([L.orc_float_to_half(float(v)) for v in xs], dtype=np.uint16).reshape(np.shape(x))


def quantize_rows(half_bits: np.ndarray, t: int) -> np.ndarray:
    """binary16 rows (uint16 [..., d]) -> rows in format t (uint8 [..., row_bytes]),
    one 32-value block at a time with the oracle's quantiser."""
    L = lib()
    h = np.ascontiguousarray(half_bits, dtype=np.uint16)
    d = h.shape[-1]
    blocks = h.reshape(-1, 32)
    bb = {F16: 64, Q4_0: 18, Q8_0: 34}[t]
    out = np.empty((blocks.shape[0], bb), np.uint8)
    for i in range(blocks.shape[0]):
        if L.orc_quantize_block(t, _ptr(blocks[i]), _ptr(out[i])) != bb:
            raise ValueError("orc_quantize_block")
    return out.reshape(*h.shape[:-1], d // 32 * bb)


def group_offset(t: int, role: int, r: int, i: int, d: int = 256) -> int:
    """Byte offset, inside its 16-row group, of byte i of the row stored in
    group row r (-1 outside the layout)."""
    return int(lib().orc_group_offset(t, role, d, r, i))


def scatter(pool: np.ndarray, n_blocks: int, hkv: int, page_size: int, t: int, role: int,
            rows: np.ndarray, row_seq: np.ndarray, row_pos: np.ndarray, table: np.ndarray,
            d: int = 256) -> int:
    """Write packed rows [n][hkv][rb] of format t into a pool of the given role
    (uint8, modified in place)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rp = np.ascontiguousarray(row_pos, dtype=np.int32)
    tab = np.ascontiguousarray(table, dtype=np.int32)
    assert pool.flags.c_contiguous and pool.dtype == np.uint8
    return int(lib().orc_scatter(_ptr(pool), n_blocks, hkv, page_size, t, role, d, _ptr(rows),
                                 _ptr(rs), _ptr(rp), rows.shape[0], _ptr(tab), tab.shape[1],
                                 tab.shape[0]))


class Cache:
    """A paged K/V cache held in host memory, built by the oracle's own scatter."""

    def __init__(self, seq_lens, n_qtok, page_size, n_blocks, k_type, v_type, table,
                 k_pool, v_pool, hq=24, hkv=4, d=256):
        self.seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.table = np.ascontiguousarray(table, dtype=np.int32)
        self.k_pool = k_pool
        self.v_pool = v_pool
        self.s = _Cache(len(self.seq_lens), n_qtok, hq, hkv, d, page_size, n_blocks, k_type, v_type,
                        self.table.ctypes.data, self.table.shape[1], self.seq_lens.ctypes.data,
                        k_pool.ctypes.data, v_pool.ctypes.data)

    @classmethod
    def from_workload(cls, w, table=None, n_blocks=None):
        """Scatter the workload's logical rows into fresh pools."""
        tab = w.table if table is None else table
        nb = w.n_blocks if n_blocks is None else n_blocks
        hkv = w.k_rows.shape[1]
        rbk, rbv = w.k_rows.shape[2], w.v_rows.shape[2]
        kp = np.zeros(nb * hkv * w.page_size * rbk, np.uint8)
        vp = np.zeros(nb * hkv * w.page_size * rbv, np.uint8)
        rs, rp = w.row_seq, w.row_pos
        d = w.q.shape[3]
        rc = scatter(kp, nb, hkv, w.page_size, w.k_type, ROLE_K, w.k_rows, rs, rp, tab, d)
        rc |= scatter(vp, nb, hkv, w.page_size, w.v_type, ROLE_V, w.v_rows, rs, rp, tab, d)
        if rc:
            raise ValueError(f"scatter rc={rc}")
        return cls(w.seq_lens, w.n_qtok, w.page_size, nb, w.k_type, w.v_type, tab, kp, vp,
                   hq=w.q.shape[2], hkv=hkv, d=w.q.shape[3])


def decode(cache: Cache, q: np.ndarray, scale: float, select: np.ndarray | None = None,
           n_threads: int = 1):
    """out float64 [n_seq][n_qtok][hq][d], lse float64 [n_seq][n_qtok][hq].

    `select` (bool [n_seq][hq]) limits the work to chosen (seq, q-head) pairs;
    unselected outputs are NaN."""
    s = cache.s
    q = np.ascontiguousarray(q, dtype=np.float32)
    assert q.shape == (s.n_seq, s.n_qtok, s.hq, s.d), q.shape
    out = np.full((s.n_seq, s.n_qtok, s.hq, s.d), np.nan)
    lse = np.full((s.n_seq, s.n_qtok, s.hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib().orc_decode(C.byref(s), _ptr(q), scale, None if sel is None else _ptr(sel),
                          _ptr(out), _ptr(lse), n_threads)
    if rc:
        raise OracleError(rc)
    return out, lse


class OracleError(RuntimeError):
    pass


def attend_range(cache: Cache, q: np.ndarray, scale: float, s: int, t: int, h: int, j0: int, j1: int):
    """Partial (o normalised, m, l) over keys [j0, j1) for query (s, t, h)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    o = np.empty(cache.s.d, np.float64)
    m, l = C.c_double(), C.c_double()
    rc = lib().orc_attend_range(C.byref(cache.s), _ptr(q), scale, s, t, h, j0, j1, _ptr(o),
                                C.byref(m), C.byref(l))
    if rc:
        raise OracleError(rc)
    return o, m.value, l.value


def merge(ms, ls, os_):
    """Merge partials; returns (out float64 [d], lse)."""
    m = np.ascontiguousarray(ms, dtype=np.float64)
    l = np.ascontiguousarray(ls, dtype=np.float64)
    o = np.ascontiguousarray(os_, dtype=np.float64)
    d = o.shape[-1]
    out = np.empty(d, np.float64)
    lse = C.c_double()
    lib().orc_merge(len(m), _ptr(m), _ptr(l), _ptr(o), d, _ptr(out), C.byref(lse))
    return out, lse.value


def decode_workload(w, n_threads: int = 1, select=None, table=None, n_blocks=None):
    """Oracle output for a `workloads.Workload` (float64 out, lse)."""
    cache = Cache.from_workload(w, table, n_blocks)
    return decode(cache, w.q, w.scale, select, n_threads)
