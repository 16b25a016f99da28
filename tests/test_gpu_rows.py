"""Row tiles: decode of 9 to 96 query tokens against the float64 oracle.

The fork gives paged K/V of up to 96 query tokens the decode kernel's row tiles
(llama.cpp fork PR #2, the commit on KV-streaming ubatches of more than 8
tokens); the computation is the causal verify decode of the narrower widths.
These tests cover widths 9 to 96 with the shortest legal sequence (L = n_qtok),
ragged lengths over several row tiles, key tiles and pieces, all nine K x V
format pairs, inputs that reach the online-softmax rescale, the paged ==
contiguous bit-identity, batches of more than 128 sequences and the device
length guard.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, assert_lse_close, device_cache, run_decode, to_dev
from paged_kv_gqa_11_gb300 import PA_ERR_BOUNDS, PA_OK, pa_decode_plan

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
F16, Q4, Q8 = W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0
NAMES = {F16: "f16", Q4: "q4_0", Q8: "q8_0"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_gqa_11_gb300 import _build
    _build.build()
    oracle.build()


def _check(w, what):
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what=what)
    assert_lse_close(gl, ol, what=what)
    return go, gl


# (name, lengths, page size, K, V, n_qtok)
SMALL = [
    ("q8q4-96-min", [700, 96, 130], 16, Q8, Q4, 96),
    ("q4-17", [1000, 17, 300], 64, Q4, Q4, 17),
    ("q8-33", [2000, 33], 256, Q8, Q8, 33),
    ("f16-65", [500, 65], 32, F16, F16, 65),
    ("f16k-q8v-9", [9, 300, 1234], 16, F16, Q8, 9),
    ("q8q4-65-long", [5000], 256, Q8, Q4, 65),
    ("q4k-f16v-22-ps48", [130, 129], 48, Q4, F16, 22),
    ("q8-96-one-row-tile-edge", [150, 96], 16, Q8, Q8, 21),  # 126 rows: one row tile, 2 padding rows
    ("q8-43-two-row-tiles", [3000, 43], 16, Q8, Q8, 43),     # 258 rows: three row tiles, the last two rows
    ("q4k-q8v-64-full-tiles", [200, 64, 1100], 32, Q4, Q8, 64),  # 384 rows: three full row tiles, no padding
]


@pytest.mark.parametrize("name,lens,ps,kt,vt,nq", SMALL, ids=[c[0] for c in SMALL])
def test_row_tile_parity(name, lens, ps, kt, vt, nq):
    _check(W.make_workload(name, 500 + len(name), lens, ps, kt, vt, nq, "shuffled"), name)


PAIRS = [(kt, vt) for kt in (F16, Q4, Q8) for vt in (F16, Q4, Q8)]


@pytest.mark.parametrize("kt,vt", PAIRS, ids=[f"k{NAMES[k]}-v{NAMES[v]}" for k, v in PAIRS])
def test_row_tiles_every_format_pair(kt, vt):
    w = W.make_workload(f"rows-pair-{kt}-{vt}", 600 + 10 * kt + vt, [900, 40, 2100], 16, kt, vt, 20, "shuffled")
    _check(w, f"k{NAMES[kt]} v{NAMES[vt]}")


STRESS = [(kind, kt, vt, nq) for kind in W.STRESS_KINDS for kt, vt in ((Q8, Q4), (F16, F16), (Q4, Q4))
          for nq in (12, 40)]


@pytest.mark.parametrize("kind,kt,vt,nq", STRESS,
                         ids=[f"{c[0]}-k{NAMES[c[1]]}-v{NAMES[c[2]]}-{c[3]}tok" for c in STRESS])
def test_row_tiles_stress(kind, kt, vt, nq):
    w = W.stress_workload(kind, 700 + 10 * kt + vt + nq, [9000, 700, nq], 64, kt, vt, nq)
    _check(w, f"{kind} k{NAMES[kt]} v{NAMES[vt]} nq{nq}")


def test_row_tiles_paged_equals_contiguous_and_repeats():
    """Row tiles through any page size and placement give the bit-identical
    result of an identity table, and repeats are identical (TensorFold #1156,
    Design / Kernels: paging changes where rows are read, not how keys sum)."""
    base = W.make_workload("rows-inv", 81, [3000, 129, 1025], 16, Q8, Q4, 30, "identity")
    ref_o, ref_l = run_decode(base)
    for ps in (16, 48, 256):
        lists = W.interleaved_blocks(base.seq_lens, ps)
        n = sum(len(l) for l in lists)
        perm = np.random.default_rng(ps).permutation(n)
        tab = W.table_from_lists([[int(perm[b]) for b in l] for l in lists])
        w = W.Workload("rows-inv", base.seq_lens, 30, ps, n, Q8, Q4, tab, base.k_rows, base.v_rows, base.q)
        c, t = device_cache(w)
        for _ in range(2):
            o, l = run_decode(w, c, t)
            assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l), ps


def test_row_tiles_plan():
    """A row tile takes the 64-key tiles its last row sees: earlier row tiles
    of a long verify batch stop short of the newest keys."""
    w = W.make_workload("rows-plan", 82, [5000, 300], 16, Q8, Q8, 96, "shuffled")
    c, _ = device_cache(w)
    plan = pa_decode_plan(c.pool, w.seq_lens, 96)
    tiles = 0
    for L in w.seq_lens:
        for rt in range(5):  # 576 rows = five row tiles of 128
            t_last = min(95, (128 * (rt + 1) - 1) // 6)
            tiles += (int(L) - 96 + t_last + 1 + 63) // 64
    assert plan["tiles"] == tiles * W.HKV and plan["tile_keys"] == 64


def test_row_tiles_sub_batches():
    rng = np.random.default_rng(83)
    lens = rng.integers(10, 300, size=140).astype(np.int32)
    _check(W.make_workload("rows-sub", 83, lens, 16, Q4, Q8, 10, "shuffled"), "rows sub-batches")


def test_row_tiles_device_lengths_are_checked():
    w = W.make_workload("rows-guard", 84, [600, 80, 2000], 16, Q8, Q4, 20, "shuffled")
    cache, tab = device_cache(w)
    oo, ol = oracle.decode_workload(w)
    q = to_dev(w.q)
    for bad_s, bad_len in ((0, 616), (2, 1 << 30)):
        dev = w.seq_lens.copy()
        dev[bad_s] = bad_len
        out, lse = cache.decode(q, tab, to_dev(dev), w.seq_lens, 20, w.scale)
        torch.cuda.synchronize()
        assert cache.check() == PA_ERR_BOUNDS
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert (o[bad_s] == 0).all() and np.isneginf(l[bad_s]).all()
        for s in range(w.n_seq):
            if s != bad_s:
                assert_close(o[s], oo[s], what=f"unaffected sequence {s}")
    out, lse = cache.decode(q, tab, to_dev(w.seq_lens), w.seq_lens, 20, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == PA_OK


def test_row_tiles_bounds_guard_reports_and_stays_finite():
    """A table entry outside the pool is never dereferenced: its rows read as
    zeros, PA_ERR_BOUNDS is reported, the output stays finite and a sequence
    that does not use the entry is unaffected (lucebox PR #555, Validation)."""
    w = W.make_workload("rows-bnd", 85, [700, 90, 1500], 16, Q8, Q4, 20, "shuffled")
    cache, _ = device_cache(w)
    bad = w.table.copy()
    bad[0, 5] = w.n_blocks + 1000
    bad[2, 40] = -7
    out, lse = cache.decode(to_dev(w.q), to_dev(bad), to_dev(w.seq_lens), w.seq_lens, 20, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == PA_ERR_BOUNDS
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    oo, ol = oracle.decode_workload(w)
    assert_close(out.cpu().numpy()[1], oo[1], what="unaffected sequence")
    assert_lse_close(lse.cpu().numpy()[1], ol[1], what="unaffected sequence")


@pytest.mark.parametrize("ctx,nq", [(4096, 17), (16384, 65), (4096, 96)])
def test_row_tile_workloads_sampled(ctx, nq):
    """The bench's row-tile workloads (one sequence, Q8_0 K / Q4_0 V): every
    query token of two query heads of different KV heads."""
    w = W.rows_workload(ctx, nq)
    go, gl = run_decode(w)
    sel = np.zeros((1, W.HQ), bool)
    sel[0, [1, 20]] = True
    oo, ol = oracle.decode_workload(w, n_threads=THREADS, select=sel)
    for h in (1, 20):
        assert_close(go[0, :, h], oo[0, :, h], what=f"rows {ctx} {nq} h{h}")
        assert_lse_close(gl[0, :, h], ol[0, :, h], what=f"rows {ctx} {nq} h{h}")
