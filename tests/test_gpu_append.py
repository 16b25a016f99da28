"""Append/scatter kernel: byte-exact against the oracle's host scatter, and a
resident multi-step append equals a one-shot upload (colibri PR #372:
"a multi-step decode that stays token-identical to the non-resident path")."""
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
