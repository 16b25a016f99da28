"""Append/scatter kernel: byte-exact against the oracle's host scatter, and a
resident multi-step append equals a one-shot upload (colibri PR #372: a
resident cache advanced step by step must match the path that uploads
everything)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import device_cache, to_dev
from paged_kv_gqa_11_gb300 import PA_ERR_BOUNDS, PA_OK
from paged_kv_gqa_11_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu


def oracle_pools(w):
    c = oracle.Cache.from_workload(w)
    return c.k_pool, c.v_pool


CASES = [
    ("f16-ps16", [300, 17], 16, W.TYPE_F16, W.TYPE_F16, "shuffled"),
    ("q4-ps32", [40, 3], 32, W.TYPE_Q4_0, W.TYPE_Q4_0, "shuffled"),
    ("q8-ps48", [500, 96, 1], 48, W.TYPE_Q8_0, W.TYPE_Q8_0, "interleaved"),
    ("mixed-ps256", [700], 256, W.TYPE_Q8_0, W.TYPE_Q4_0, "shuffled"),
]


@pytest.mark.parametrize("name,lens,ps,kt,vt,layout", CASES, ids=[c[0] for c in CASES])
def test_append_matches_host_scatter(name, lens, ps, kt, vt, layout):
    w = W.make_workload(name, 50, lens, ps, kt, vt, 1, layout)
    c, _ = device_cache(w)
    ko, vo = oracle_pools(w)
    assert np.array_equal(c.k_pool.cpu().numpy(), ko)
    assert np.array_equal(c.v_pool.cpu().numpy(), vo)


def test_multistep_append_equals_one_shot():
    """Warm each sequence, then append one row per sequence per step (the
    resident decode pattern): the pools end byte-identical to one upload."""
    w = W.make_workload("steps", 51, [90, 33, 64], 16, W.TYPE_Q4_0, W.TYPE_Q4_0, 1, "shuffled")
    one, _ = device_cache(w)
    inc = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type)
    tab = to_dev(w.table)
    order = np.lexsort((w.row_seq, w.row_pos))  # step by position, all sequences per step
    warm = 16
    first = order[w.row_pos[order] < warm]
    rest = order[w.row_pos[order] >= warm]
    chunks = [first] + [rest[w.row_pos[rest] == p] for p in np.unique(w.row_pos[rest])]
    for idx in chunks:
        inc.append(to_dev(w.k_rows[idx]), to_dev(w.v_rows[idx]), to_dev(w.row_seq[idx]), to_dev(w.row_pos[idx]), tab)
    assert inc.check() == PA_OK
    assert torch.equal(inc.k_pool, one.k_pool) and torch.equal(inc.v_pool, one.v_pool)


def test_append_bounds_guard():
    """Rows whose table entry lies outside the pool are skipped and reported;
    nothing else is written."""
    w = W.make_workload("b", 52, [40], 16, W.TYPE_F16, W.TYPE_F16, 1, "identity")
    bad = w.table.copy()
    bad[0, 1] = w.n_blocks + 7          # rows 16..31 point outside the pool
    c = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type)
    c.append(to_dev(w.k_rows), to_dev(w.v_rows), to_dev(w.row_seq), to_dev(w.row_pos), to_dev(bad))
    assert c.check() == PA_ERR_BOUNDS
    good = w.table.copy()
    keep = (w.row_pos < 16) | (w.row_pos >= 32)
    ref = W.Workload("b", w.seq_lens, 1, 16, w.n_blocks, w.k_type, w.v_type, good, w.k_rows, w.v_rows, w.q)
    ko, vo = oracle_pools(ref)
    # expected: oracle scatter of the rows that had a valid entry only
    ko2 = np.zeros_like(ko)
    vo2 = np.zeros_like(vo)
    oracle.scatter(ko2, w.n_blocks, 4, 16, w.k_type, oracle.ROLE_K, w.k_rows[keep], w.row_seq[keep], w.row_pos[keep], good)
    oracle.scatter(vo2, w.n_blocks, 4, 16, w.v_type, oracle.ROLE_V, w.v_rows[keep], w.row_seq[keep], w.row_pos[keep], good)
    assert np.array_equal(c.k_pool.cpu().numpy(), ko2)
    assert np.array_equal(c.v_pool.cpu().numpy(), vo2)


# ------------------------------------------------------------------ quantise on append

def _rows_f16(rng, n):
    """binary16 sources [n][4][256] with planted edge blocks: all zero, ties in
    magnitude, products that land exactly on .5 (d = 1 blocks), tiny values."""
    x = rng.standard_normal((n, 4, 256)).astype(np.float32)
    x[0, 0, :32] = 0.0
    x[0, 1, :32] = np.linspace(-2, 2, 32)          # -2 and +2: a tie in magnitude
    x[1, 2, :32] = 0.0
    x[1, 2, 0] = 127.0                             # Q8_0 d = 1: q = x exactly
    x[1, 2, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]
    x[1, 3, :32] = 0.0
    x[1, 3, 0] = -8.0                              # Q4_0 d = 1
    x[1, 3, 1:9] = [-7.5, 6.5, 7.0, 7.5, -0.5, 0.5, 0.25, -8.0]
    x[2, 0, :32] *= 1e-5                           # scales in the fp16 subnormal range
    return x.astype(np.float16).view(np.uint16)


QCASES = [("q4_0", W.TYPE_Q4_0, W.TYPE_Q4_0), ("q8_0", W.TYPE_Q8_0, W.TYPE_Q8_0),
          ("f16", W.TYPE_F16, W.TYPE_F16), ("q8k-q4v", W.TYPE_Q8_0, W.TYPE_Q4_0)]


@pytest.mark.parametrize("name,kt,vt", QCASES, ids=[c[0] for c in QCASES])
def test_quantise_on_append_matches_oracle(name, kt, vt):
    """fp16 rows quantised by the append kernel give, byte for byte, the pools
    of the oracle's quantiser followed by the oracle's scatter."""
    w = W.make_workload(name, 60, [100, 33, 16, 48], 16, kt, vt, 1, "shuffled")
    rng = np.random.default_rng(61)
    n = int(w.row_seq.shape[0])
    hk, hv = _rows_f16(rng, n), _rows_f16(rng, n)
    ref = W.Workload(name, w.seq_lens, 1, w.page_size, w.n_blocks, kt, vt, w.table,
                     oracle.quantize_rows(hk, kt), oracle.quantize_rows(hv, vt), w.q)
    ko, vo = oracle_pools(ref)
    c = PagedKVCache(w.n_blocks, w.page_size, kt, vt)
    c.append_f16(to_dev(hk), to_dev(hv), to_dev(w.row_seq), to_dev(w.row_pos), to_dev(w.table))
    assert c.check() == PA_OK
    assert np.array_equal(c.k_pool.cpu().numpy(), ko)
    assert np.array_equal(c.v_pool.cpu().numpy(), vo)


def test_quantise_on_append_large_sampled():
    """The many-sequence workload's shape (64 sequences, lognormal lengths,
    Q8_0 K with Q4_0 V) quantised on append; sampled rows against the oracle's
    quantiser, read back through the documented pool layout."""
    base = W.config(5, variant="b")
    rng = np.random.default_rng(62)
    n = int(base.row_seq.shape[0])
    hk = rng.standard_normal((n, 4, 256)).astype(np.float16).view(np.uint16)
    hv = rng.standard_normal((n, 4, 256)).astype(np.float16).view(np.uint16)
    kt, vt = W.TYPE_Q8_0, W.TYPE_Q4_0
    c = PagedKVCache(base.n_blocks, base.page_size, kt, vt)
    c.append_f16(to_dev(hk), to_dev(hv), to_dev(base.row_seq), to_dev(base.row_pos), to_dev(base.table))
    assert c.check() == PA_OK
    kp, vp = c.k_pool.cpu().numpy(), c.v_pool.cpu().numpy()
    pick = rng.choice(n, 64, replace=False)
    for t, role, pool, src in ((kt, oracle.ROLE_K, kp, hk), (vt, oracle.ROLE_V, vp, hv)):
        rb = oracle.row_bytes(t)
        offs = np.array([[oracle.group_offset(t, role, r, i) for i in range(rb)] for r in range(16)])
        want = oracle.quantize_rows(src[pick], t)
        for k, i in enumerate(pick):
            s, pos = int(base.row_seq[i]), int(base.row_pos[i])
            blk = int(base.table[s, pos // base.page_size])
            slot = pos % base.page_size
            for h in range(4):
                grp = ((blk * 4 + h) * base.page_size + slot // 16 * 16) * rb
                got = pool[grp + offs[slot % 16]]
                assert np.array_equal(got, want[k, h]), (t, i, h)
