"""The seeded input generators make what they claim (CPU).

The stress inputs must really drive a decoder's running maximum up after the
first keys, by more than the margin after which the decoders rescale; this is
checked with the oracle's own dequantisation, on the CPU, so that the GPU
parity tests that use them are known to reach the rescale paths.
"""
import numpy as np
import pytest

import oracle
import workloads as W

LAZY_NATS = 8.0 * np.log(2.0)  # the decoders raise their reference maximum past 2^8


def _logits(w, s, h, t):
    """Scaled logits of query (s, t, h) over its visible keys, float64."""
    g = h // W.GQA
    off = int(w.seq_offsets[s])
    L = int(w.seq_lens[s])
    vis = L - w.n_qtok + t + 1
    k = oracle.dequant_rows(w.k_rows[off:off + vis, g], w.k_type)
    return w.scale * (k @ w.q[s, t, h].astype(np.float64))


def _raises(z, tile):
    """How often a lazy running maximum (raised only past LAZY_NATS, checked
    per tile of `tile` keys) is raised while it already holds weight."""
    m, n = -np.inf, 0
    for a in range(0, len(z), tile):
        mx = z[a:a + tile].max()
        if mx > m + LAZY_NATS:
            n += np.isfinite(m)
            m = mx
    return n


@pytest.mark.parametrize("kind", ["rising", "late", "bigq"])
@pytest.mark.parametrize("kt", [W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0])
def test_stress_inputs_raise_the_running_max(kind, kt):
    w = W.stress_workload(kind, 5, [6000, 40], 16, kt, W.TYPE_Q8_0, 2)
    z = _logits(w, 0, 0, w.n_qtok - 1)
    assert z[64:].max() - z[:64].max() > LAZY_NATS + 1.0, (kind, z[:64].max(), z[64:].max())
    assert _raises(z, 16) >= 1 and _raises(z, 64) >= 1


def test_stress_scales_have_zero_and_subnormal_blocks():
    w = W.stress_workload("scales", 6, [500], 16, W.TYPE_Q8_0, W.TYPE_Q4_0, 1)
    for rows, bb in ((w.k_rows, 34), (w.v_rows, 18)):
        d = rows.reshape(-1, bb)[:, :2].copy().view("<f2").astype(np.float64).ravel()
        assert (d == 0).any()
        sub = (d != 0) & (np.abs(d) < 2.0 ** -14)
        assert sub.any() and (np.abs(d) > 2.0 ** -14).any()


def test_stress_bigq_is_binary16_exact():
    w = W.stress_workload("bigq", 7, [100], 16, W.TYPE_F16, W.TYPE_F16, 3)
    assert np.array_equal(w.q.astype(np.float16).astype(np.float32), w.q)
    assert w.q.std() > 10


def test_stress_layout_matches_make_workload_tables():
    """Same lengths and page size: the same table shape and a permutation of
    the same blocks as make_workload's shuffled layout."""
    a = W.stress_workload("late", 8, [300, 17, 64], 16, W.TYPE_Q4_0, W.TYPE_Q4_0, 1)
    b = W.make_workload("x", 8, [300, 17, 64], 16, W.TYPE_Q4_0, W.TYPE_Q4_0, 1, "shuffled")
    assert a.table.shape == b.table.shape and a.n_blocks == b.n_blocks
    assert sorted(a.table[a.table >= 0].tolist()) == list(range(a.n_blocks))
