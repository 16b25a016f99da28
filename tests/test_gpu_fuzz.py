"""Seeded random shapes against the float64 oracle: every query-token width
from one to 96 (both kernel families), all three storage formats for K and
for V independently, page sizes 16 to 256, sequence lengths from n_qtok (the
shortest legal) to a few thousand, shuffled or interleaved pools.  Each case
compares every output row and its lse with the oracle (TensorFold #1156,
Verification: the float64 bound holds for any placement).
"""
import os

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import assert_close, assert_lse_close, run_decode

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
TYPES = (W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0)
N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_gqa_11_gb300 import _build
    _build.build()
    oracle.build()


def _case(i):
    rng = np.random.default_rng(9000 + i)
    nq = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8])) if i % 2 == 0 else int(rng.integers(9, 97))
    n_seq = int(rng.integers(1, 5))
    lens = [int(nq if rng.random() < 0.2 else rng.integers(nq, 3000)) for _ in range(n_seq)]
    ps = int(rng.choice([16, 32, 48, 64, 256]))
    kt, vt = (int(x) for x in rng.choice(TYPES, size=2))
    layout = "shuffled" if rng.random() < 0.7 else "interleaved"
    return f"fuzz{i}-nq{nq}-ps{ps}-k{kt}-v{vt}", lens, ps, kt, vt, nq, layout


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    name, lens, ps, kt, vt, nq, layout = _case(i)
    w = W.make_workload(name, 9000 + i, lens, ps, kt, vt, nq, layout)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(go, oo, what=name)
    assert_lse_close(gl, ol, what=name)
