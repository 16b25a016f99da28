"""Decode parity: the CUDA path against the float64 oracle, element by element,
plus the bit-identity gates (paged == contiguous for any page size, repeats
identical) and the controls that must fail (TensorFold #1156, Verification)."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, assert_lse_close, device_cache, run_decode, to_dev
from paged_kv_gqa_11_gb300 import (PA_ERR_BOUNDS, PA_ERR_TIMEOUT, PA_OK, _build, pa_decode_plan,
                                   pa_selftest_wait_timeout)
from paged_kv_gqa_11_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


F16, Q4, Q8 = W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0

# (name, lengths, page size, K type, V type, n_qtok, layout): several tiles,
# ragged tails, page sizes that do and do not divide the 64-key tile.
SMALL = [
    ("f16-1tok", [300], 16, F16, F16, 1, "shuffled"),
    ("q4-edges", [1, 63, 64, 65, 129], 16, Q4, Q4, 1, "shuffled"),
    ("q8-ps32-2tok", [200, 7], 32, Q8, Q8, 2, "shuffled"),
    ("q8-masked-4tok", [513, 64, 4], 256, Q8, Q8, 4, "shuffled"),
    ("f16-ps48-3tok", [1000, 130], 48, F16, F16, 3, "interleaved"),
    ("q4-ps80-4tok", [777], 80, Q4, Q4, 4, "shuffled"),
    ("q4-mix-2tok", [2048, 333, 17, 4096], 64, Q4, Q4, 2, "shuffled"),
    ("q8-min-len", [1, 2, 3], 16, Q8, Q8, 1, "shuffled"),
    ("f16-min-len-4tok", [4, 5, 6, 67], 16, F16, F16, 4, "shuffled"),
    ("q4-5tok", [300, 77, 5], 16, Q4, Q4, 5, "shuffled"),
    ("f16-6tok", [200, 7, 6], 32, F16, F16, 6, "interleaved"),
    ("q8-7tok", [130, 8, 65], 16, Q8, Q8, 7, "shuffled"),
    ("q8k-q4v-8tok", [500, 9, 64], 256, Q8, Q4, 8, "shuffled"),
]


@pytest.mark.parametrize("name,lens,ps,kt,vt,nq,layout", SMALL, ids=[c[0] for c in SMALL])
def test_small_parity(name, lens, ps, kt, vt, nq, layout):
    w = W.make_workload(name, 200 + len(name), lens, ps, kt, vt, nq, layout)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what=name)
    assert_lse_close(gl, ol, what=name)


PAIRS = [(kt, vt) for kt in (F16, Q4, Q8) for vt in (F16, Q4, Q8)]
NAMES = {F16: "f16", Q4: "q4_0", Q8: "q8_0"}


@pytest.mark.parametrize("kt,vt", PAIRS, ids=[f"k{NAMES[k]}-v{NAMES[v]}" for k, v in PAIRS])
@pytest.mark.parametrize("nq", [1, 3])
def test_every_format_pair(kt, vt, nq):
    """All nine K x V format pairs (Q8_0 K with Q4_0 V is the production
    pair of lucebox PR #555), one and three query tokens, ragged lengths with
    partial last tiles and a multi-piece sequence."""
    w = W.make_workload(f"pair-{kt}-{vt}", 300 + 10 * kt + vt, [2100, 77, 16, 600], 16, kt, vt, nq, "shuffled")
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what=f"k{kt} v{vt} nq{nq}")
    assert_lse_close(gl, ol, what=f"k{kt} v{vt} nq{nq}")


def test_many_short_sequences():
    """More tiles than CTAs: CTAs walk many whole segments and restage Q."""
    rng = np.random.default_rng(9)
    lens = rng.integers(1, 300, size=200)
    lens = np.maximum(lens, 2)
    w = W.make_workload("many-short", 9, lens, 16, Q8, Q8, 2, "shuffled")
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="many-short")
    assert_lse_close(gl, ol, what="many-short")


def test_config1_tiny():
    w = W.config(1)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w)
    assert_close(go, oo, what="config1")
    assert_lse_close(gl, ol, what="config1")


def test_config2_uniform():
    w = W.config(2)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="config2")
    assert_lse_close(gl, ol, what="config2")


@pytest.fixture(scope="module")
def ragged():
    w = W.config(3)
    cache, tab = device_cache(w)
    go, gl = run_decode(w, cache, tab)
    return w, go, gl


def test_config3_ragged_full(ragged):
    """Every (sequence, query head) row of the ragged batch."""
    w, go, gl = ragged
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="config3")
    assert_lse_close(gl, ol, what="config3")


def test_config3_paged_equals_contiguous(ragged):
    """Same rows through an identity table padded to 131072 slots per
    sequence: bit-identical output (TensorFold #1156: paged == contiguous)."""
    w, go, gl = ragged
    wc = W.config(3, variant="contiguous")
    co, cl = run_decode(wc)
    assert np.array_equal(go, co) and np.array_equal(gl, cl)


def test_page_size_invariance_and_repeats():
    """Any page size and placement, same rows: bit-identical; three repeats
    identical."""
    base = W.make_workload("inv", 77, [3000, 129, 1025], 16, Q4, Q4, 3, "identity")
    ref_o, ref_l = run_decode(base)
    for ps in (16, 32, 48, 64, 80, 256):
        lists = W.interleaved_blocks(base.seq_lens, ps)
        n = sum(len(l) for l in lists)
        perm = np.random.default_rng(ps).permutation(n)
        tab = W.table_from_lists([[int(perm[b]) for b in l] for l in lists])
        w = W.Workload("inv", base.seq_lens, 3, ps, n, Q4, Q4, tab, base.k_rows, base.v_rows, base.q)
        c, t = device_cache(w)
        for _ in range(3):
            o, l = run_decode(w, c, t)
            assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l), ps


@pytest.mark.parametrize("nq", [1, 2, 3, 4, 5, 6, 7, 8])
def test_config4_verify(nq):
    """The verify workload at one to four tokens, and at five to eight (the
    wider verify batches the fork's decode kernel later took); every row."""
    w = W.config(4, n_qtok=nq)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what=f"config4 nq{nq}")
    assert_lse_close(gl, ol, what=f"config4 nq{nq}")


def test_config5a_long_f16_full():
    w = W.config(5, variant="a")
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="config5a")
    assert_lse_close(gl, ol, what="config5a")


def test_config5b_many_full():
    w = W.config(5, variant="b")
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="config5b")
    assert_lse_close(gl, ol, what="config5b")


def test_fully_masked_split_is_finite():
    """L = 513 with 4 query tokens: the tile holding key 512 is visible only to
    the last token; the merge must give finite output that matches."""
    w = W.make_workload("mask", 88, [513], 256, Q8, Q8, 4, "shuffled")
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w)
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    assert_close(go, oo, what="masked")


def test_controls_are_red():
    """Two controls that must fail the comparison (TensorFold #1156,
    Verification): a table whose pages are swapped while the data stays in
    place, and a planted wrong row."""
    w = W.make_workload("ctl", 99, [700, 300], 16, Q4, Q4, 1, "shuffled")
    oo, _ = oracle.decode_workload(w)
    cache, tab = device_cache(w)
    good, _ = run_decode(w, cache, tab)
    assert_close(good, oo, what="control baseline")
    # Attention is a function of the set of (k, v) rows, so the swap moves a
    # page between sequences: sequence 0 then reads sequence 1's rows.
    swapped = w.table.copy()
    swapped[0, 2], swapped[1, 5] = w.table[1, 5], w.table[0, 2]
    bad, _ = run_decode(w, cache, to_dev(swapped))
    with pytest.raises(AssertionError):
        assert_close(bad, oo, what="swapped table")
    # planted row: overwrite K of position 100 (seq 1) with position 0's row
    planted = w.k_rows.copy()
    off = int(w.seq_offsets[1])
    planted[off + 100] = planted[off + 0]
    wp = W.Workload("ctl", w.seq_lens, 1, 16, w.n_blocks, Q4, Q4, w.table, planted, w.v_rows, w.q)
    bad2, _ = run_decode(wp)
    with pytest.raises(AssertionError):
        assert_close(bad2, oo, what="planted row")


def test_bounds_guard_reports_and_stays_finite():
    w = W.make_workload("bnd", 5, [300, 80], 16, Q8, Q8, 1, "shuffled")
    cache, tab = device_cache(w)
    bad = w.table.copy()
    bad[0, 3] = w.n_blocks + 1000
    q = to_dev(w.q)
    out, lse = cache.decode(q, to_dev(bad), to_dev(w.seq_lens), w.seq_lens, 1, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == PA_ERR_BOUNDS
    assert torch.isfinite(out).all()
    # sequence 1 does not touch the bad entry: still exact
    oo, _ = oracle.decode_workload(w)
    assert_close(out.cpu().numpy()[1], oo[1], what="unaffected sequence")


@pytest.mark.parametrize("nq", [1, 3])
def test_device_lengths_are_checked(nq):
    """The decode walks the host copy of the lengths; a device length that
    differs from it (longer by a page, past the table's capacity, negative,
    shorter by one key) gives zeros and lse -inf for that sequence and
    PA_ERR_BOUNDS, and reads nothing outside the sequence's table row (lucebox
    PR #555, Validation: guards against corrupt block-table bounds).  The
    other sequences stay exact; the long one is split over many CTAs."""
    w = W.make_workload("lenguard", 61, [300, 80, 1000], 16, Q8, Q8, nq, "shuffled")
    cache, tab = device_cache(w)
    oo, ol = oracle.decode_workload(w)
    cap = tab.shape[1] * w.page_size
    q = to_dev(w.q)
    for bad_s, bad_len in ((0, 316), (2, 1 << 30), (1, -5), (1, 79), (2, cap + 16)):
        dev = w.seq_lens.copy()
        dev[bad_s] = bad_len
        out, lse = cache.decode(q, tab, to_dev(dev), w.seq_lens, nq, w.scale)
        torch.cuda.synchronize()
        assert cache.check() == PA_ERR_BOUNDS, (bad_s, bad_len)
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert (o[bad_s] == 0).all() and np.isneginf(l[bad_s]).all(), (bad_s, bad_len)
        for s in range(w.n_seq):
            if s != bad_s:
                assert_close(o[s], oo[s], what=f"unaffected sequence {s}")
                assert_lse_close(l[s], ol[s], what=f"unaffected sequence {s}")
    # and the same call with agreeing lengths is clean
    out, lse = cache.decode(q, tab, to_dev(w.seq_lens), w.seq_lens, nq, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == PA_OK
    assert_close(out.cpu().numpy(), oo, what="agreeing lengths")


def test_large_batch_runs_in_sub_batches():
    """More sequences than one launch takes (128): the library runs
    consecutive sub-batches that share the workspace; the result matches the
    oracle and a repeat is bit-identical.  The separate split / merge passes
    refuse such a batch."""
    rng = np.random.default_rng(41)
    lens = rng.integers(3, 400, size=300).astype(np.int32)
    lens[7] = 5000
    w = W.make_workload("subbatch", 41, lens, 16, Q4, Q8, 3, "shuffled")
    cache, tab = device_cache(w)
    go, gl = run_decode(w, cache, tab)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="sub-batches")
    assert_lse_close(gl, ol, what="sub-batches")
    go2, gl2 = run_decode(w, cache, tab)
    assert np.array_equal(go, go2) and np.array_equal(gl, gl2)
    from paged_kv_gqa_11_gb300 import PA_ERR_UNSUPPORTED, pa_decode
    q, sl = to_dev(w.q), to_dev(w.seq_lens)
    out = torch.empty_like(q)
    ws = cache.workspace(w.n_seq, w.n_qtok)
    rc = pa_decode(cache.pool, q, cache.k_pool, cache.v_pool, tab, tab.shape[1], sl, w.seq_lens, w.n_seq, 3, W.HQ,
                   w.scale, out, None, ws, ws.numel(), cache.err, check=False, passes="split")
    assert rc == PA_ERR_UNSUPPORTED


def test_bounded_wait_expires_with_status():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert pa_selftest_wait_timeout(2000, err) == PA_OK
    torch.cuda.synchronize()
    assert int(err.item()) == PA_ERR_TIMEOUT


def test_plan_covers_every_tile():
    """One query token: 16-key tiles of all four KV heads (one segment per
    sequence); more tokens: 64-key tiles of one head (four per sequence)."""
    w = W.config(3)
    c = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for nq, keys, segs in ((1, 16, 1), (2, 64, W.HKV)):
        plan = pa_decode_plan(c.pool, w.seq_lens, nq)
        tiles = int(sum((L + keys - 1) // keys for L in w.seq_lens)) * segs
        assert plan["tiles"] == tiles and plan["tile_keys"] == keys, (nq, plan)
        assert 0 < plan["ctas"] <= tiles
        assert plan["ctas"] % sms == 0 or plan["ctas"] == tiles
        assert plan["partials"] >= w.n_seq * segs


def _weighted_pieces(lens, keys, segs, ctas, w):
    """Pieces of the CTA cut over a cost where a tile costs 1 and a segment's
    first tile w more, by brute force: CTA i starts at the smallest x whose
    cost of tiles [0, x) reaches floor(i * total / ctas)."""
    n = [(L + keys - 1) // keys for L in lens for _ in range(segs)]
    starts = np.cumsum([0] + n[:-1])
    T = int(sum(n))
    cost = np.arange(T + 1) + w * np.searchsorted(starts, np.arange(T + 1), side="left")
    total = T + w * len(n)
    cut = [int(np.argmax(cost >= (i * total) // ctas)) for i in range(ctas)] + [T]
    assert all(b > a for a, b in zip(cut, cut[1:]))
    owner = np.searchsorted(cut, np.arange(T), side="right") - 1
    return sum(int(owner[s + k - 1]) - int(owner[s]) + 1 for s, k in zip(starts, n))


def test_plan_weights_segment_starts():
    """Two to eight query tokens: the CTA ranges are cut at equal cost with a
    segment's first tile weighing two tiles more, so ranges that hold segment
    starts get fewer tiles; one token keeps equal tile counts."""
    c = PagedKVCache(8, 256, W.TYPE_Q8_0, W.TYPE_Q8_0)
    mixed = [9000] * 3 + [130] * 100  # many segment starts
    for lens, nq, keys, segs, w in ((W.VERIFY_LENGTHS, 1, 16, 1, 0), (W.VERIFY_LENGTHS, 3, 64, W.HKV, 2),
                                    (W.VERIFY_LENGTHS, 8, 64, W.HKV, 2), (mixed, 3, 64, W.HKV, 2)):
        plan = pa_decode_plan(c.pool, lens, nq)
        assert plan["partials"] == _weighted_pieces(lens, keys, segs, plan["ctas"], w), (nq, plan)
    assert plan["partials"] != _weighted_pieces(mixed, 64, W.HKV, plan["ctas"], 0)


def test_prefix_fork_with_copy_on_write():
    """Sequence A (100 rows) is forked into B by sharing its blocks.  B's
    partly filled last page is copied on write before B appends 20 rows; A
    then appends 10 other rows into its own, now unshared, last page.  Both
    decode like the oracle on their logical rows, and the copy is byte-exact."""
    from paged_kv_gqa_11_gb300 import pa_copy_blocks
    ps, kt, vt = 16, Q8, Q4
    rng = np.random.default_rng(91)
    c = PagedKVCache(32, ps, kt, vt)
    pool = c.pool
    rows_k = W.random_rows(rng, 130, kt)
    rows_v = W.random_rows(rng, 130, vt)
    a_pre, a_new, b_new = slice(0, 100), slice(100, 110), slice(110, 130)
    hA = pool.alloc(7)
    tA = [pool.block_index(h)[1] for h in hA]

    def put(table_row, k, v, positions):
        n = len(positions)
        tab = to_dev(np.array([table_row + [-1] * (8 - len(table_row))], np.int32))
        c.append(to_dev(k), to_dev(v), to_dev(np.zeros(n, np.int32)), to_dev(np.array(positions, np.int32)), tab)
        assert c.check() == PA_OK

    put(tA, rows_k[a_pre], rows_v[a_pre], list(range(100)))
    # fork: B shares A's blocks
    assert pool.share(hA) == PA_OK and pool.refcount(hA[6]) == (PA_OK, 2)
    rc, (hB6,), copies = pool.cow([hA[6]])
    assert rc == PA_OK and len(copies) == 1 and copies[0][0] == tA[6]
    pa_copy_blocks(pool, c.k_pool, c.v_pool, to_dev(np.array([copies[0][0]], np.int32)),
                   to_dev(np.array([copies[0][1]], np.int32)), 1, c.err)
    assert c.check() == PA_OK
    kb = c.k_pool.view(32, -1)
    vb = c.v_pool.view(32, -1)
    assert torch.equal(kb[copies[0][1]], kb[tA[6]]) and torch.equal(vb[copies[0][1]], vb[tA[6]])
    hB7 = pool.alloc(1)[0]
    tB = tA[:6] + [copies[0][1], pool.block_index(hB7)[1]]
    put(tB, rows_k[b_new], rows_v[b_new], list(range(100, 120)))
    # A's last page is now held once: cow keeps it
    rc, (hA6,), none = pool.cow([hA[6]])
    assert rc == PA_OK and hA6 == hA[6] and none == []
    put(tA, rows_k[a_new], rows_v[a_new], list(range(100, 110)))
    table = np.full((2, 8), -1, np.int32)
    table[0, :7] = tA
    table[1, :8] = tB
    lens = np.array([110, 120], np.int32)
    q = rng.standard_normal((2, 1, W.HQ, W.D), dtype=np.float32)
    out, lse = c.decode(to_dev(q), to_dev(table), to_dev(lens), lens, 1)
    c.raise_on_error()
    # the oracle sees each sequence's logical rows through its own private layout
    ref = W.Workload("fork", lens, 1, ps, 15, kt, vt,
                     W.table_from_lists([list(range(7)), list(range(7, 15))]),
                     np.concatenate([rows_k[a_pre], rows_k[a_new], rows_k[a_pre], rows_k[b_new]]),
                     np.concatenate([rows_v[a_pre], rows_v[a_new], rows_v[a_pre], rows_v[b_new]]), q)
    oo, ol = oracle.decode_workload(ref, n_threads=THREADS)
    assert_close(out.cpu().numpy(), oo, what="fork")
    assert_lse_close(lse.cpu().numpy(), ol, what="fork")
    # dropping B's references frees only B's private pages
    free0 = pool.free_count()
    assert pool.release(hA[:6] + [hB6, hB7]) == PA_OK and pool.free_count() == free0 + 2


def test_shared_prefix_batch_full():
    """Eight sequences sharing a prompt's pages: every row matches the oracle,
    and sharing leaves results equal to a private copy of the prefix (the
    contiguous layout)."""
    w = W.shared_prefix(n_seq=8, prefix=4096, own=300)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what="shared prefix")
    assert_lse_close(gl, ol, what="shared prefix")
    co, cl = run_decode(w.contiguous())
    assert np.array_equal(go, co) and np.array_equal(gl, cl)


def test_append_then_decode_back_to_back():
    """Decode steps as a server runs them: each step appends one new row per
    sequence and decodes at once on the same stream, with no host
    synchronisation in between.  The decode is launched as a programmatic
    dependent of the append and must still see every appended row: each
    step's output matches the oracle on the rows present at that step."""
    import dataclasses
    steps = 6
    lens_final = np.array([160, 97, 33], np.int32)
    w = W.make_workload("back-to-back", 909, lens_final, 16, Q4, Q4, 1, "shuffled")
    base = lens_final - steps

    def rows(sel):
        return (to_dev(w.k_rows[sel]), to_dev(w.v_rows[sel]), to_dev(w.row_seq[sel]), to_dev(w.row_pos[sel]))

    cache = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type)
    tab = to_dev(w.table)
    pos_limit = base[w.row_seq]
    cache.append(*rows(w.row_pos < pos_limit), tab)
    step_rows = [rows(w.row_pos == pos_limit + t) for t in range(steps)]  # uploaded before the loop
    q = to_dev(w.q)
    lens_dev = [to_dev(base + t + 1) for t in range(steps)]
    torch.cuda.synchronize()
    results = []
    for t in range(steps):
        cache.append(*step_rows[t], tab)
        lens = base + t + 1
        out, lse = cache.decode(q, tab, lens_dev[t], lens, 1, w.scale)
        results.append((lens, out, lse))
    torch.cuda.synchronize()
    assert cache.check() == PA_OK
    for lens, out, lse in results:
        keep = w.row_pos < lens[w.row_seq]
        wt = dataclasses.replace(w, seq_lens=lens.astype(np.int32), k_rows=w.k_rows[keep], v_rows=w.v_rows[keep])
        oo, ol = oracle.decode_workload(wt)
        assert_close(out.cpu().numpy(), oo, what=f"lengths {lens.tolist()}")
        assert_lse_close(lse.cpu().numpy(), ol, what=f"lengths {lens.tolist()}")


def test_split_then_merge_equals_decode():
    """pa_decode_split then pa_decode_merge on one stream is exactly
    pa_decode (same arguments and workspace, nothing in between)."""
    w = W.make_workload("split-merge", 77, [3000, 700, 41, 5000], 16, Q8, Q4, 3, "shuffled")
    cache, tab = device_cache(w)
    q = to_dev(w.q)
    sl = to_dev(w.seq_lens)
    o1, l1 = cache.decode(q, tab, sl, w.seq_lens, w.n_qtok, w.scale)
    o2 = torch.full_like(o1, float("nan"))
    l2 = torch.full_like(l1, float("nan"))
    cache.decode(q, tab, sl, w.seq_lens, w.n_qtok, w.scale, out=o2, lse=l2, passes="split")
    cache.decode(q, tab, sl, w.seq_lens, w.n_qtok, w.scale, out=o2, lse=l2, passes="merge")
    torch.cuda.synchronize()
    assert cache.check() == PA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_reads_inputs_written_just_before():
    """Q and the lengths are produced by kernels launched on the stream right
    before the decode, with no synchronisation: the decode (a programmatic
    dependent launch) still reads the values they write."""
    w = W.make_workload("fresh-inputs", 78, [900, 64, 2000], 16, Q4, Q4, 1, "shuffled")
    cache, tab = device_cache(w)
    q_half = to_dev(w.q * 0.5)
    sl_src = to_dev(w.seq_lens - 1)
    torch.cuda.synchronize()
    q = q_half * 2.0          # a kernel writing q
    sl = sl_src + 1           # a kernel writing the device lengths
    out, lse = cache.decode(q, tab, sl, w.seq_lens, w.n_qtok, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == PA_OK
    oo, ol = oracle.decode_workload(w)
    assert_close(out.cpu().numpy(), oo, what="fresh inputs")
    assert_lse_close(lse.cpu().numpy(), ol, what="fresh inputs")
