"""Pins for the float64 oracle: it is checked against things other than itself.

Each `pin_*` function raises AssertionError when the oracle is wrong.  The
test functions run them against the real oracle; `test_planted_mistakes`
recompiles copies of the oracle with one plausible mistake each and checks
that some pin turns red.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D, HQ, HKV = W.D, W.HQ, W.HKV


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def workload_from_sources(lengths, ps, kt, vt, n_qtok, k_src, v_src, q, layout="shuffled", seed=0):
    """A workload whose rows are the given float sources (encoded per type)."""
    base = W.make_workload("pin", seed, [1], 16, W.TYPE_F16, W.TYPE_F16, 1, "identity")
    lengths = np.asarray(lengths, np.int32)
    rng = np.random.default_rng(seed + 1000)
    lists = W.interleaved_blocks(lengths, ps)
    n_pages = sum(len(l) for l in lists)
    if layout == "shuffled":
        perm = rng.permutation(n_pages)
        lists = [[int(perm[b]) for b in l] for l in lists]
    table = W.table_from_lists(lists)
    del base
    return W.Workload("pin", lengths, n_qtok, ps, n_pages, kt, vt, table,
                      W.encode_rows(np.asarray(k_src, np.float32), kt),
                      W.encode_rows(np.asarray(v_src, np.float32), vt),
                      np.asarray(q, np.float32), W.SCALE)


# ------------------------------------------------------------------ formats

def pin_half_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _f16_bits(x):
    return int(np.float16(x).view(np.uint16))


def pin_q8_0_hand_block():
    # d = 0.5, q_i = 8*i - 127 clipped, a second block with d = -2 and q = +-127
    blk0 = bytearray(np.uint16(_f16_bits(0.5)).tobytes())
    q0 = [max(-127, min(127, 8 * i - 127)) for i in range(32)]
    blk0 += bytes([v & 0xFF for v in q0])
    blk1 = bytearray(np.uint16(_f16_bits(-2.0)).tobytes())
    q1 = [127 if i % 2 == 0 else -127 for i in range(32)]
    blk1 += bytes([v & 0xFF for v in q1])
    row = bytes(blk0 + blk1) + bytes(34 * 6)  # remaining blocks: d = 0, q = 0
    got = oracle.dequant_rows(np.frombuffer(row, np.uint8)[None], W.TYPE_Q8_0)[0]
    want = np.zeros(256)
    want[:32] = [0.5 * v for v in q0]
    want[32:64] = [-2.0 * v for v in q1]
    assert np.array_equal(got, want), np.nonzero(got != want)


def pin_q4_0_hand_block():
    # byte j: low nibble j%16, high nibble 15-(j%16).  Element j = (j-8)*d,
    # element j+16 = (7-j)*d.
    d = 0.25
    blk = bytearray(np.uint16(_f16_bits(d)).tobytes())
    blk += bytes([(j & 0xF) | ((15 - j) << 4) for j in range(16)])
    # second block: all nibbles 0 (value -8 d) with d = 3 ; third: all 15 with d = -1.5
    blk2 = bytes(np.uint16(_f16_bits(3.0)).tobytes()) + bytes(16)
    blk3 = bytes(np.uint16(_f16_bits(-1.5)).tobytes()) + bytes([0xFF] * 16)
    row = bytes(blk) + blk2 + blk3 + bytes(18 * 5)
    got = oracle.dequant_rows(np.frombuffer(row, np.uint8)[None], W.TYPE_Q4_0)[0]
    want = np.zeros(256)
    for j in range(16):
        want[j] = (j - 8) * d
        want[j + 16] = (7 - j) * d
    want[32:64] = -8 * 3.0
    want[64:96] = 7 * -1.5
    want[96:] = 0.0  # d = 0 in the remaining blocks
    assert np.array_equal(got, want), np.nonzero(got != want)


def pin_subnormal_and_negative_scales():
    # A Q8_0 block whose scale is the smallest subnormal fp16 (2^-24).
    row = bytearray(34 * 8)
    row[0:2] = np.uint16(1).tobytes()
    row[2] = 100
    row[3] = 0x9C  # -100
    got = oracle.dequant_rows(np.frombuffer(bytes(row), np.uint8)[None], W.TYPE_Q8_0)[0]
    assert got[0] == 100 * 2.0 ** -24 and got[1] == -100 * 2.0 ** -24


def pin_capacity_table():
    """The Q4_0 block size from the pages' capacity numbers: MiB * 2^20 over
    tokens x heads x (K+V) x blocks-per-row gives bytes per 32-value block."""
    g = _golden("capacity_lucebox.json")
    for mib, tokens in ((g["paged_one_layer_mib"], g["live_tokens"]),
                        (g["padded_one_layer_mib"], g["padded_slots"])):
        per_block = mib * 2 ** 20 / (tokens * g["n_kv_heads"] * 2 * (g["head_dim"] // 32))
        assert per_block == 18.0, per_block
    assert oracle.row_bytes(W.TYPE_Q4_0) == 18 * 8
    assert round(g["padded_one_layer_mib"] / g["paged_one_layer_mib"], 2) == g["ratio_printed"]


def pin_rdna4_bandwidth():
    """Q8_0 (34 B) K + Q4_0 (18 B) V bytes per call over the printed time give
    the printed ~590 GB/s at 131k with one query token."""
    g = _golden("rdna4_percall.json")
    us = g["us_per_call"]["131072"][0]
    kv = 131072 * g["n_kv_heads"] * (oracle.row_bytes(W.TYPE_Q8_0) + oracle.row_bytes(W.TYPE_Q4_0))
    gbps = kv / (us * 1e-6) / 1e9
    assert abs(gbps - g["gbps_printed_1_2_tokens"]) / g["gbps_printed_1_2_tokens"] < 0.01, gbps


def pin_quantiser_roundtrip():
    """Generator bytes dequantised by the oracle are within half a step of the
    float sources (catches a wrong offset, sign or nibble order)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256), dtype=np.float32)
    # Q8_0 rounds to the nearest of 255 symmetric steps: half a step.  Q4_0
    # has 16 levels -8..7 times d = -max/8, so the side opposite the block's
    # largest element clamps at 7 and may be off by one full step.
    for t, steps, bound in ((W.TYPE_Q8_0, 127.0, 0.5), (W.TYPE_Q4_0, 8.0, 1.0)):
        rows = W.encode_rows(x, t)
        y = oracle.dequant_rows(rows, t)
        amax = np.abs(x.reshape(-1, 32)).max(1)
        step = (amax / steps).repeat(32).reshape(x.shape)
        # plus the fp16 rounding of the scale (relative 2^-11 of |x|)
        err = np.abs(y - x)
        assert (err <= bound * step * 1.002 + np.abs(x) * 2.0 ** -10 + 1e-7).all(), err.max()
        assert np.mean(err <= 0.5 * step * 1.002 + np.abs(x) * 2.0 ** -10 + 1e-7) > 0.97
    rows = W.encode_rows(x, W.TYPE_F16)
    assert np.array_equal(oracle.dequant_rows(rows, W.TYPE_F16), x.astype(np.float16).astype(np.float64))


# ------------------------------------------------------------------ attention closed forms

def _onehot_q(n_seq, n_qtok, dim, value):
    q = np.zeros((n_seq, n_qtok, HQ, D), np.float32)
    q[..., dim] = value
    return q


def pin_one_key():
    """One cached key: out = v exactly, lse = scale*q.k; with q = 16 e_3 and
    k_3 = 1.75 the logit is exactly 1.75."""
    for kt in (W.TYPE_F16, W.TYPE_Q8_0, W.TYPE_Q4_0):
        rng = np.random.default_rng(kt)
        k = np.zeros((1, HKV, D), np.float32)
        k[..., 3] = 1.75
        if kt == W.TYPE_Q4_0:
            k[..., 5] = -2.0  # block max -> d = 0.25, so 1.75 = (15-8)*0.25 exactly
        if kt == W.TYPE_Q8_0:
            k[..., 5] = 127 / 16  # block max -> d = 1/16, so 1.75 = 28 * d exactly
        v = rng.standard_normal((1, HKV, D), dtype=np.float32)
        w = workload_from_sources([1], 16, kt, kt, 1, k, v, _onehot_q(1, 1, 3, 16.0))
        out, lse = oracle.decode_workload(w)
        vd = oracle.dequant_rows(w.v_rows, kt)[0]
        for h in range(HQ):
            assert np.array_equal(out[0, 0, h], vd[h // 6]), (kt, h)
            assert lse[0, 0, h] == 1.75, (kt, h, lse[0, 0, h])


def pin_identical_keys_and_zero_query():
    """All keys equal: uniform weights, out = mean of the visible values and
    lse = z + ln(n).  A zero query gives the same with z = 0."""
    rng = np.random.default_rng(11)
    L = 37
    k = np.tile(rng.standard_normal((1, HKV, D), dtype=np.float32), (L, 1, 1))
    v = rng.standard_normal((L, HKV, D), dtype=np.float32)
    q = rng.standard_normal((1, 1, HQ, D), dtype=np.float32)
    w = workload_from_sources([L], 16, W.TYPE_F16, W.TYPE_F16, 1, k, v, q)
    out, lse = oracle.decode_workload(w)
    vd = oracle.dequant_rows(w.v_rows, W.TYPE_F16)
    kd = oracle.dequant_rows(w.k_rows[:1], W.TYPE_F16)[0]
    for h in range(HQ):
        g = h // 6
        assert np.allclose(out[0, 0, h], vd[:, g].mean(0), rtol=1e-12, atol=1e-14)
        z = W.SCALE * float(np.dot(q[0, 0, h].astype(np.float64), kd[g]))
        assert abs(lse[0, 0, h] - (z + np.log(L))) < 1e-12
    w0 = w.with_q(np.zeros_like(q), 1)
    out0, lse0 = oracle.decode_workload(w0)
    assert np.allclose(out0[0, 0], vd.mean(0).repeat(6, axis=0), rtol=1e-12, atol=1e-14)
    assert np.allclose(lse0, np.log(L), rtol=0, atol=1e-13)


def pin_gqa_mapping():
    """V constant per KV head g (value (g+1)/2): query head h must return
    (h//6 + 1)/2 -- contiguous groups of six."""
    rng = np.random.default_rng(12)
    L = 50
    k = rng.standard_normal((L, HKV, D), dtype=np.float32)
    v = np.zeros((L, HKV, D), np.float32)
    for g in range(HKV):
        v[:, g, :] = (g + 1) / 2
    q = rng.standard_normal((2, 1, HQ, D), dtype=np.float32)
    w = workload_from_sources([L // 2, L // 2], 32, W.TYPE_Q8_0, W.TYPE_F16, 1, k, v, q)
    out, _ = oracle.decode_workload(w)
    for h in range(HQ):
        assert np.allclose(out[:, 0, h], (h // 6 + 1) / 2, rtol=1e-13), h


def pin_causal_verify():
    """n_qtok = 4, L = 9, identical keys, v_j = j: query t sees keys 0..5+t,
    so out = (5+t)/2 and lse = z + ln(6+t)."""
    L, nq = 9, 4
    k = np.ones((L, HKV, D), np.float32) * 0.5
    v = np.zeros((L, HKV, D), np.float32)
    for j in range(L):
        v[j] = j
    q = np.zeros((1, nq, HQ, D), np.float32)
    q[..., 0] = 2.0  # z = (1/16) * 2 * 0.5 = 1/16
    w = workload_from_sources([L], 16, W.TYPE_F16, W.TYPE_F16, nq, k, v, q)
    out, lse = oracle.decode_workload(w)
    for t in range(nq):
        assert np.allclose(out[0, t], (5 + t) / 2, rtol=1e-13), (t, out[0, t, 0, 0])
        assert np.allclose(lse[0, t], 1 / 16 + np.log(6 + t), rtol=0, atol=1e-13)


def pin_dominant_key():
    """One key with logit 80 above the rest: out = that key's value (to
    e^-80), found through a shuffled table across pages."""
    L = 40
    for jstar in (0, 17, 39):
        rng = np.random.default_rng(jstar)
        k = np.zeros((L, HKV, D), np.float32)
        k[jstar, :, 0] = 8.0
        v = rng.standard_normal((L, HKV, D), dtype=np.float32)
        q = _onehot_q(1, 1, 0, 160.0)
        w = workload_from_sources([L], 16, W.TYPE_F16, W.TYPE_Q8_0, 1, k, v, q)
        out, lse = oracle.decode_workload(w)
        vd = oracle.dequant_rows(w.v_rows, W.TYPE_Q8_0)
        for h in range(HQ):
            assert np.allclose(out[0, 0, h], vd[jstar, h // 6], rtol=1e-12, atol=1e-12)
            assert abs(lse[0, 0, h] - 80.0) < 1e-12


def _dense_reference(w):
    """numpy/scipy brute force over the logical rows (no pool, no table)."""
    kd = oracle.dequant_rows(w.k_rows, w.k_type)   # [T][HKV][D]
    vd = oracle.dequant_rows(w.v_rows, w.v_type)
    off = w.seq_offsets
    out = np.zeros(w.q.shape, np.float64)
    lse = np.zeros(w.q.shape[:3], np.float64)
    for s in range(w.n_seq):
        L = int(w.seq_lens[s])
        ks, vs = kd[off[s]:off[s] + L], vd[off[s]:off[s] + L]
        for t in range(w.n_qtok):
            vis = L - w.n_qtok + t + 1
            for h in range(HQ):
                g = h // (HQ // HKV)
                if vis <= 0:
                    lse[s, t, h] = -np.inf
                    continue
                z = w.scale * (ks[:vis, g] @ w.q[s, t, h].astype(np.float64))
                p = scipy.special.softmax(z)
                out[s, t, h] = p @ vs[:vis, g]
                lse[s, t, h] = scipy.special.logsumexp(z)
    return out, lse


def pin_dense_brute_force():
    cases = [([7, 1, 20], 16, W.TYPE_F16, W.TYPE_F16, 1),
             ([33, 16], 16, W.TYPE_Q4_0, W.TYPE_Q4_0, 2),
             ([5, 40], 32, W.TYPE_Q8_0, W.TYPE_Q8_0, 4),
             ([18, 50], 48, W.TYPE_Q8_0, W.TYPE_Q4_0, 3),
             ([20, 37], 16, W.TYPE_Q8_0, W.TYPE_Q4_0, 20),   # row-tile widths, L = n_qtok included
             ([96, 130], 16, W.TYPE_F16, W.TYPE_Q8_0, 96)]
    for i, (lens, ps, kt, vt, nq) in enumerate(cases):
        w = W.make_workload("bf", 100 + i, lens, ps, kt, vt, nq, "shuffled")
        out, lse = oracle.decode_workload(w)
        ro, rl = _dense_reference(w)
        assert np.allclose(out, ro, rtol=1e-11, atol=1e-13), (i, np.abs(out - ro).max())
        assert np.allclose(lse, rl, rtol=1e-12, atol=1e-12), (i, np.abs(lse - rl).max())


def pin_placement_and_page_size_invariance():
    """Shuffled placement and any page size give bit-identical output
    (TensorFold #1156: paged == contiguous for any page size)."""
    base = W.make_workload("inv", 21, [45, 16, 70], 16, W.TYPE_Q4_0, W.TYPE_Q4_0, 2, "identity")
    ref_out, ref_lse = oracle.decode_workload(base)
    for ps in (16, 32, 48, 128, 256):
        for layout in ("identity", "shuffled"):
            rng = np.random.default_rng(ps)
            lists = W.interleaved_blocks(base.seq_lens, ps)
            n = sum(len(l) for l in lists)
            if layout == "shuffled":
                perm = rng.permutation(n + 5)  # pool with holes
                lists = [[int(perm[b]) for b in l] for l in lists]
            w = W.Workload("inv", base.seq_lens, base.n_qtok, ps, n + 5, base.k_type, base.v_type,
                           W.table_from_lists(lists), base.k_rows, base.v_rows, base.q)
            out, lse = oracle.decode_workload(w)
            assert np.array_equal(out, ref_out), (ps, layout)
            assert np.array_equal(lse, ref_lse), (ps, layout)


def pin_split_merge():
    """Any partition of the visible keys, merged by log-sum-exp, equals the
    unsplit softmax (llama.cpp fork PR #2, LSE commit), over 1024 random
    splittings (the pages' count for their merge oracle), including empty
    (fully masked) parts."""
    w = W.make_workload("sm", 31, [70, 9], 16, W.TYPE_Q8_0, W.TYPE_Q4_0, 3, "shuffled")
    cache = oracle.Cache.from_workload(w)
    full_out, full_lse = oracle.decode(cache, w.q, w.scale)
    rng = np.random.default_rng(7)
    for case in range(1024):
        s = int(rng.integers(0, 2))
        t = int(rng.integers(0, 3))
        h = int(rng.integers(0, HQ))
        L = int(w.seq_lens[s])
        k = int(rng.integers(1, 8))
        cuts = np.sort(rng.integers(0, L + 1, size=k))
        bounds = [0] + cuts.tolist() + [L + 3]  # the last part reaches past L: masked keys
        parts = [oracle.attend_range(cache, w.q, w.scale, s, t, h, a, b)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        o, lse = oracle.merge([p[1] for p in parts], [p[2] for p in parts], [p[0] for p in parts])
        assert np.allclose(o, full_out[s, t, h], rtol=1e-12, atol=1e-14), case
        assert abs(lse - full_lse[s, t, h]) < 1e-12, case


def pin_fully_masked_part():
    """A part holding only masked keys has m = -inf, l = 0; merging it in
    changes nothing and an all-masked merge gives 0 (not NaN) and -inf."""
    w = W.make_workload("fm", 41, [513], 256, W.TYPE_Q8_0, W.TYPE_Q8_0, 4, "shuffled")
    cache = oracle.Cache.from_workload(w)
    o, m, l = oracle.attend_range(cache, w.q, w.scale, 0, 0, 0, 512, 513)  # t=0 sees keys <= 509
    assert m == -np.inf and l == 0.0 and not np.any(o)
    o3, m3, l3 = oracle.attend_range(cache, w.q, w.scale, 0, 3, 0, 512, 513)  # t=3 sees key 512
    assert np.isfinite(m3) and l3 == 1.0
    out, lse = oracle.merge([m, m], [l, l], [o, o])
    assert lse == -np.inf and np.array_equal(out, np.zeros(D))


# ------------------------------------------------------------------ quantise on append

def pin_float_to_half_vs_numpy():
    """fp32 -> fp16 rounding (nearest, ties to even) against numpy's own
    binary16 conversion: random values over the whole range, exact ties,
    subnormals, overflow and signed zeros."""
    rng = np.random.default_rng(17)
    parts = [rng.standard_normal(4000).astype(np.float32) * np.float32(2.0) ** rng.integers(-30, 18, 4000)]
    # exact halfway points between neighbouring binary16 values (ties)
    h = rng.integers(0, 0x7bff, 2000).astype(np.uint16)
    a = h.view(np.float16).astype(np.float32)
    b = (h + 1).astype(np.uint16).view(np.float16).astype(np.float32)
    parts.append(((a.astype(np.float64) + b.astype(np.float64)) / 2).astype(np.float32))
    parts.append(np.array([0.0, -0.0, 65504, 65519.99, 65520, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                           1.5 * 2.0 ** -25, 2.0 ** -26, 6.1e-5, 6.097e-5], np.float32))
    x = np.concatenate(parts)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.float_to_half(x), ref)


def _h(vals):
    return np.asarray(vals, np.float32).astype(np.float16).view(np.uint16)


def pin_quantiser_closed_forms():
    """Blocks whose quantisation is known in closed form."""
    # Q8_0: x = k/8, amax = 127/8 -> d = 1/8 exactly, q = k exactly
    k = np.arange(-127, 128, 8)[:32].astype(np.float32)
    k[0] = -127
    out = oracle.quantize_rows(_h(k / 8), W.TYPE_Q8_0)
    assert out[0] == 0x00 and out[1] == 0x30  # fp16(0.125)
    assert np.array_equal(out[2:].view(np.int8), k.astype(np.int8))
    # Q8_0 rounds half away from zero: d = 1, x = +-2.5 -> +-3, +-0.5 -> +-1
    x = np.zeros(32, np.float32)
    x[:5] = [127, 2.5, -2.5, 0.5, -0.5]
    q = oracle.quantize_rows(_h(x), W.TYPE_Q8_0)[2:].view(np.int8)
    assert list(q[:5]) == [127, 3, -3, 1, -1] and not q[5:].any()
    # Q4_0: largest magnitude -2 (first on ties) -> d = 0.25; x = (q - 8) / 4 -> q
    qs = np.arange(32) % 16
    x = (qs - 8) / 4.0
    x[1], x[17] = -2.0, 2.0  # a tie in magnitude: the first (-2) sets d = +0.25; +2 clamps to 15
    out = oracle.quantize_rows(_h(x), W.TYPE_Q4_0)
    assert out[0] == 0x00 and out[1] == 0x34  # fp16(0.25)
    nib = np.concatenate([out[2:] & 15, out[2:] >> 4])
    want = qs.copy()
    want[1], want[17] = 0, 15
    assert np.array_equal(nib, want)
    # Q4_0 with a positive extreme: d = -m/8 < 0, the extreme maps to q = 0
    x = np.zeros(32, np.float32)
    x[3] = 4.0
    out = oracle.quantize_rows(_h(x), W.TYPE_Q4_0)
    assert out[0] == 0x00 and out[1] == 0xb8  # fp16(-0.5)
    nib = np.concatenate([out[2:] & 15, out[2:] >> 4])
    assert nib[3] == 0 and (np.delete(nib, 3) == 8).all()
    # all-zero blocks
    z = np.zeros(32, np.uint16)
    assert np.array_equal(oracle.quantize_rows(z, W.TYPE_Q8_0), np.zeros(34, np.uint8))
    zq4 = oracle.quantize_rows(z, W.TYPE_Q4_0)
    assert zq4[1] == 0x80 and zq4[0] == 0 and (zq4[2:] == 0x88).all()  # d = 0 / -8 = -0.0
    # F16 is a copy
    r = np.random.default_rng(3).integers(0, 0x7c00, 256).astype(np.uint16)
    assert np.array_equal(oracle.quantize_rows(r, W.TYPE_F16).view(np.uint16), r)


def pin_quantiser_error_bounds():
    """Dequantised values lie within half a step (Q8_0) or one step (Q4_0) of
    the input, plus what storing the scale in fp16 adds (|q| <= 128 times a
    relative 2^-11 of the step: 1/16 of a step), most within half a step."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    h = _h(x)
    xf = h.view(np.float16).astype(np.float64)
    for t, steps, bound in ((W.TYPE_Q8_0, 127.0, 0.5), (W.TYPE_Q4_0, 8.0, 1.0)):
        deq = oracle.dequant_rows(oracle.quantize_rows(h, t), t)
        amax = np.abs(xf.reshape(-1, 32)).max(axis=1)
        step = (amax / steps).repeat(32).reshape(xf.shape)
        err = np.abs(deq - xf)
        assert (err <= (bound + 1 / 16) * step + 1e-12).all(), t
        assert (err <= 0.5 * step * (1 + 1e-3) + 1e-12).mean() > 0.97, t


# ------------------------------------------------------------------ pool layout

# Offsets worked out by hand from the written layout definition (pa.h, "Pool
# layout"): (format, role, group row r, byte i of the row) -> byte in the group.
LAYOUT_FIXTURES = [
    (W.TYPE_Q4_0, oracle.ROLE_K, 0, 0, 0),        # scale of block 0, row 0
    (W.TYPE_Q4_0, oracle.ROLE_K, 3, 37, 53),      # block 2 scale, high byte: 2*(3*8+2)+1
    (W.TYPE_Q4_0, oracle.ROLE_K, 3, 38, 656),     # quant chunk 2 -> 2^3 = 1: 256 + (24+1)*16
    (W.TYPE_Q4_0, oracle.ROLE_K, 13, 143, 1967),  # chunk 7 -> 7^5 = 2: 256 + (104+2)*16 + 15
    (W.TYPE_Q4_0, oracle.ROLE_V, 11, 90, 158),    # block 5 scale: 128 + 16 + 8 + 4 + 2
    (W.TYPE_Q4_0, oracle.ROLE_V, 6, 1, 49),       # block 0 scale, high byte: 16*3 + 1
    (W.TYPE_Q4_0, oracle.ROLE_V, 2, 18, 24),      # block 1 scale: 16*1 + 8*1
    (W.TYPE_Q4_0, oracle.ROLE_V, 9, 1, 7),        # block 0 scale, high byte: 4*1 + 2*1 + 1
    (W.TYPE_Q8_0, oracle.ROLE_K, 2, 35, 35),      # block 1 scale, high byte: 2*(16+1)+1
    (W.TYPE_Q8_0, oracle.ROLE_K, 2, 52, 784),     # quant 48 = chunk 3 -> 3^2 = 1: 256 + 33*16
    (W.TYPE_Q8_0, oracle.ROLE_K, 9, 271, 2799),   # chunk 15 -> 15^1 = 14: 256 + 158*16 + 15
    (W.TYPE_Q8_0, oracle.ROLE_V, 13, 102, 110),   # block 3 scale: 64 + 16*2 + 8 + 4 + 2
    (W.TYPE_F16, oracle.ROLE_K, 5, 100, 2612),    # chunk 6 -> 6^5 = 3: (160+3)*16 + 4
    (W.TYPE_F16, oracle.ROLE_V, 15, 511, 8079),   # chunk 31 -> 31^7 = 24: (480+24)*16 + 15
]


def pin_group_layout():
    """The oracle's pool layout is the documented one: hand-worked offsets,
    every byte of a 16-row group written exactly once, and the property the
    layout exists for -- the eight rows of any 16-byte chunk column fall in
    eight different 16-byte bank groups (offset / 16 mod 8)."""
    for t, role, r, i, want in LAYOUT_FIXTURES:
        assert oracle.group_offset(t, role, r, i) == want, (t, role, r, i)
    for t in (W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0):
        rb = oracle.row_bytes(t)
        scales = 0 if t == W.TYPE_F16 else 256
        for role in (oracle.ROLE_K, oracle.ROLE_V):
            offs = np.array([[oracle.group_offset(t, role, r, i) for i in range(rb)] for r in range(16)])
            assert np.array_equal(np.sort(offs.ravel()), np.arange(16 * rb)), (t, role)
            q = offs[offs >= scales] - scales  # quant region, [16 rows][...]
            chunk_pos = (q.reshape(16, -1) // 16)
            for half in (slice(0, 8), slice(8, 16)):
                banks = chunk_pos[half] % 8
                for col in range(banks.shape[1]):
                    assert len(set(banks[:, col])) == 8, (t, role, col)
    # out-of-range arguments
    assert oracle.group_offset(W.TYPE_Q4_0, oracle.ROLE_K, 16, 0) == -1
    assert oracle.group_offset(W.TYPE_Q4_0, 2, 0, 0) == -1
    assert oracle.group_offset(W.TYPE_Q8_0, oracle.ROLE_V, 0, 272) == -1


PINS = [pin_half_all_patterns, pin_q8_0_hand_block, pin_q4_0_hand_block,
        pin_subnormal_and_negative_scales, pin_capacity_table, pin_rdna4_bandwidth,
        pin_quantiser_roundtrip, pin_one_key, pin_identical_keys_and_zero_query, pin_gqa_mapping,
        pin_causal_verify, pin_dominant_key, pin_dense_brute_force,
        pin_placement_and_page_size_invariance, pin_split_merge, pin_fully_masked_part, pin_group_layout,
        pin_float_to_half_vs_numpy, pin_quantiser_closed_forms, pin_quantiser_error_bounds]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_bounds_guard():
    """A table entry outside the pool is reported, never read."""
    w = W.make_workload("b", 3, [40], 16, W.TYPE_F16, W.TYPE_F16, 1, "shuffled")
    bad = w.table.copy()
    bad[0, 1] = w.n_blocks  # one past the end
    with pytest.raises(oracle.OracleError):
        cache = oracle.Cache(w.seq_lens, 1, 16, w.n_blocks, w.k_type, w.v_type, bad,
                             np.zeros(w.n_blocks * HKV * 16 * 512, np.uint8),
                             np.zeros(w.n_blocks * HKV * 16 * 512, np.uint8))
        oracle.decode(cache, w.q, w.scale)


# Plausible mistakes, one per variant: (name, text in the oracle, replacement).
MUTATIONS = [
    ("gqa_mod", "const int g = h / (c->hq / c->hkv);", "const int g = h % c->hkv;"),
    ("nibble_swap", "int lo = blk[2 + j] & 0x0f;\n        int hi = blk[2 + j] >> 4;",
     "int hi = blk[2 + j] & 0x0f;\n        int lo = blk[2 + j] >> 4;"),
    ("q4_no_offset", "out[32 * b + j] = (double)(lo - 8) * s;", "out[32 * b + j] = (double)(lo) * s;"),
    ("q8_unsigned", "(double)(int8_t)blk[2 + i] * s", "(double)(uint8_t)blk[2 + i] * s"),
    ("causal_off_by_one", "const long last = L - c->n_qtok + t;", "const long last = L - c->n_qtok + t + 1;"),
    ("no_scale", "z[j - j0] = scale * acc;", "z[j - j0] = acc;"),
    ("slot_off_by_one", "long slot = pos % c->page_size;", "long slot = (pos + 1) % c->page_size;"),
    ("layout_transposed",
     "const uint8_t* grp = pool + ((blk * c->hkv + g) * (long)c->page_size + slot / ORC_GROUP * ORC_GROUP) * rb;",
     "const uint8_t* grp = pool + ((blk * (long)c->page_size + slot / ORC_GROUP * ORC_GROUP) * c->hkv + g) * rb;"),
    ("layout_no_swizzle", "return 32L * nb + (r * chunks + (c ^ (r % 8))) * 16 + qi % 16;",
     "return 32L * nb + (r * chunks + c) * 16 + qi % 16;"),
    ("quant_round_even", "out[2 + i] = (uint8_t)(int8_t)roundf(v);", "out[2 + i] = (uint8_t)(int8_t)rintf(v);"),
    ("quant_q4_sign", "const float d = m / -8.0f;", "const float d = m / 8.0f;"),
    ("quant_q4_no_clamp", "q[i] = t < 15 ? t : 15;", "q[i] = t;"),
    ("half_round_up", "if (rem > half || (rem == half && (q & 1u))) ++q;", "if (rem >= half) ++q;"),
    ("v_scale_pairs", "8 * (b % 2) + 4 * (r / 8) + 2 * (r % 2) + o;", "4 * (b % 2) + 8 * (r / 8) + 2 * (r % 2) + o;"),
    ("softmax_sign", "double w = exp(z[j - j0] - m);", "double w = exp(m - z[j - j0]);"),
    ("lse_drops_max", "lse[base] = (l > 0.0) ? m + log(l) : -INFINITY;",
     "lse[base] = (l > 0.0) ? log(l) : -INFINITY;"),
    ("half_bias", "v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    ("half_subnormal", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("merge_drops_l", "double w = l[i] * exp(m[i] - M);", "double w = exp(m[i] - M);"),
    ("q_dot_transposed", "acc += (double)qv[i] * row[i];", "acc += (double)qv[i] * row[(i + 1) % d];"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes(name, old, new):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor missing: {name}"
    path = oracle.build_variant(src.replace(old, new), name)
    caught = []
    with oracle.using(path):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError, ValueError):
                caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
