"""The C-ABI library builds, loads and exports every entry point include/pa.h
declares; host-only entry points behave (no GPU needed)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import paged_kv_gqa_11_gb300 as pa
from paged_kv_gqa_11_gb300 import _build
from oracle.allocator_model import AllocatorModel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(pa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = C.CDLL(_build.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_row_bytes(lib):
    assert pa.row_bytes(pa.PA_F16) == 512
    assert pa.row_bytes(pa.PA_Q4_0) == 144
    assert pa.row_bytes(pa.PA_Q8_0) == 272
    assert pa.row_bytes(3) == 0 and pa.row_bytes(pa.PA_F16, 250) == 0


def test_pool_bytes_and_validation(lib):
    p = pa.Pool(32, 16, 4, 256, pa.PA_Q4_0, pa.PA_Q8_0)
    assert p.bytes(0) == 32 * 4 * 16 * 144
    assert p.bytes(1) == 32 * 4 * 16 * 272
    assert p.bytes(2) == 0
    for bad in [(0, 16), (4, 0)]:
        with pytest.raises(pa.PaError) as e:
            pa.Pool(bad[0], bad[1], 4, 256, pa.PA_F16)
        assert e.value.status == pa.PA_ERR_INVALID
    for bad in [(16, 256, 5), (8, 256, pa.PA_Q4_0), (24, 256, pa.PA_F16), (16, 128, pa.PA_F16)]:
        with pytest.raises(pa.PaError) as e:
            pa.Pool(8, bad[0], 4, bad[1], bad[2])  # bad type, page not whole groups, head_dim not 256
        assert e.value.status == pa.PA_ERR_UNSUPPORTED


def _random_ops(seed, n_blocks, steps):
    rng = np.random.default_rng(seed)
    lib_pool = pa.Pool(n_blocks, 16, 4, 256, pa.PA_F16)
    model = AllocatorModel(n_blocks)
    held = []
    stale = []
    for _ in range(steps):
        r = rng.random()
        if r < 0.45:
            n = int(rng.integers(0, n_blocks // 2 + 2))
            rc, hs = lib_pool.alloc_status(n)
            mrc, mhs = model.alloc(n)
            assert (rc, hs) == (mrc, mhs)
            held += hs
        elif r < 0.8 and held:
            k = int(rng.integers(1, len(held) + 1))
            idx = rng.choice(len(held), size=k, replace=False)
            rel = [held[i] for i in idx]
            if rng.random() < 0.2 and stale:
                rel.append(stale[int(rng.integers(0, len(stale)))])
            if rng.random() < 0.1:
                rel.append(rel[0])  # repeat inside one call
            rc = lib_pool.release(rel)
            assert rc == model.release(rel)
            if rc == pa.PA_OK:
                s = set(idx.tolist())
                stale += [h for i, h in enumerate(held) if i in s]
                held = [h for i, h in enumerate(held) if i not in s]
        elif r < 0.86 and held:  # share some held blocks (each share is one more reference to drop)
            k = int(rng.integers(1, min(len(held), 4) + 1))
            sh = [held[int(i)] for i in rng.choice(len(held), size=k)]
            if rng.random() < 0.2 and stale:
                sh.append(stale[-1])
            rc = lib_pool.share(sh)
            assert rc == model.share(sh)
            if rc == pa.PA_OK:
                held += sh
        elif r < 0.93 and held:  # copy-on-write of some held references
            k = int(rng.integers(1, min(len(held), 5) + 1))
            idx = sorted(rng.choice(len(held), size=k, replace=False).tolist())
            cw = [held[i] for i in idx]
            if rng.random() < 0.1 and stale:
                cw.append(stale[-1])
            got = lib_pool.cow(cw)
            assert got == model.cow(cw)
            if got[0] == pa.PA_OK:
                for i, h in zip(idx, got[1]):
                    held[i] = h
        else:
            probe = held + stale[-5:] + [(7 << 32) | (n_blocks + 3)]
            for h in probe:
                assert lib_pool.block_index(h) == model.block_index(h)
                assert lib_pool.refcount(h) == model.refcount(h)
        assert lib_pool.free_count() == model.free_count()


@pytest.mark.parametrize("seed,n_blocks", [(0, 1), (1, 7), (2, 64), (3, 333)])
def test_allocator_matches_model(lib, seed, n_blocks):
    """Handle for handle, status for status, against the plain-Python model."""
    _random_ops(seed, n_blocks, 400)


def test_allocator_oom_and_stale(lib):
    p = pa.Pool(4, 16, 4, 256, pa.PA_F16)
    hs = p.alloc(3)
    assert p.alloc_status(2)[0] == pa.PA_ERR_OOM and p.free_count() == 1
    assert p.release([hs[0]]) == pa.PA_OK
    assert p.release([hs[0]]) == pa.PA_ERR_STALE            # released already
    assert p.release([hs[1], hs[1]]) == pa.PA_ERR_STALE     # repeated: nothing released
    assert p.block_index(hs[1]) == (pa.PA_OK, 1)
    again = p.alloc(1)[0]
    assert again & 0xFFFFFFFF == 0 and again >> 32 == 2      # immediate reuse, new generation


def test_share_release_and_cow(lib):
    """Shared blocks stay live until every reference is dropped; cow swaps a
    shared block for a fresh one and lists the copy."""
    p = pa.Pool(4, 16, 4, 256, pa.PA_F16)
    a, b = p.alloc(2)
    assert p.share([a, a]) == pa.PA_OK and p.refcount(a) == (pa.PA_OK, 3)
    rc, out, copies = p.cow([a, b])
    assert rc == pa.PA_OK and out[1] == b and out[0] != a and copies == [(0, 2)]
    assert p.refcount(a) == (pa.PA_OK, 2) and p.refcount(out[0]) == (pa.PA_OK, 1)
    assert p.release([a, a, a]) == pa.PA_ERR_STALE and p.refcount(a) == (pa.PA_OK, 2)  # more than held
    assert p.release([a, a]) == pa.PA_OK and p.block_index(a)[0] == pa.PA_ERR_STALE
    assert p.alloc(1)[0] == (2 << 32) | 0  # freed at the last reference, new generation
    # not enough free blocks for the copies: nothing changes
    q = pa.Pool(2, 16, 4, 256, pa.PA_F16)
    x, y = q.alloc(2)
    q.share([x, y])
    assert q.cow([x, y])[0] == pa.PA_ERR_OOM and q.refcount(x) == (pa.PA_OK, 2) and q.free_count() == 0


def test_decode_rejects_unsupported_shapes_on_host(lib):
    """Host validation returns before any CUDA call."""
    ok = pa.Pool(8, 16, 4, 256, pa.PA_F16)
    sl = np.array([5], np.int32)
    args = dict(q=8192, k_pool=8192, v_pool=8192, block_table=8192, table_stride=8, seq_lens_dev=8192,
                seq_lens_host=sl, n_seq=1, n_qtok=1, n_q_heads=24, scale=0.0625, out=8192, lse=None,
                workspace=8192, ws_bytes=1 << 20, err=8192, stream=0, check=False)
    assert pa.pa_decode(ok, **{**args, "n_qtok": 97}) == pa.PA_ERR_UNSUPPORTED  # row tiles stop at 96
    assert pa.pa_decode(ok, **{**args, "n_qtok": 0}) == pa.PA_ERR_UNSUPPORTED
    assert pa.pa_decode(ok, **{**args, "n_qtok": 9}) == pa.PA_ERR_INVALID  # supported, but L = 5 < 9
    assert pa.pa_decode(ok, **{**args, "n_q_heads": 16}) == pa.PA_ERR_UNSUPPORTED
    assert pa.pa_decode(ok, **{**args, "q": None}) == pa.PA_ERR_INVALID
    assert pa.pa_decode(ok, **{**args, "q": 8196}) == pa.PA_ERR_INVALID   # not 16-byte aligned
    assert pa.pa_decode(ok, **{**args, "n_seq": 0}) == pa.PA_OK
    assert pa.pa_decode(ok, **{**args, "seq_lens_host": np.array([0], np.int32)}) == pa.PA_ERR_INVALID
    assert pa.pa_decode(ok, **{**args, "seq_lens_host": np.array([200], np.int32)}) == pa.PA_ERR_INVALID
    assert pa.pa_decode(ok, **{**args, "n_qtok": 2, "seq_lens_host": np.array([1], np.int32)}) == pa.PA_ERR_INVALID


def test_append_rejects_bad_arguments_on_host(lib):
    p = pa.Pool(8, 16, 4, 256, pa.PA_Q8_0)
    good = dict(k_pool=8192, v_pool=8192, k_rows=8192, v_rows=8192, row_seq=8192, row_pos=8192, n_rows=1,
                block_table=8192, table_stride=4, n_seq=1, err=8192, stream=0)
    with pytest.raises(pa.PaError) as e:
        pa.pa_append_rows(p, **{**good, "k_rows": None})
    assert e.value.status == pa.PA_ERR_INVALID
    with pytest.raises(pa.PaError) as e:
        pa.pa_append_rows(p, **{**good, "v_pool": 8200})
    assert e.value.status == pa.PA_ERR_INVALID
    pa.pa_append_rows(p, **{**good, "n_rows": 0})  # nothing to do


def test_status_strings(lib):
    for i, name in enumerate(pa.STATUS):
        assert lib.pa_status_string(i).decode() == name


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    """No fallback: a missing libpa raises instead of computing elsewhere."""
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        pa.load()
