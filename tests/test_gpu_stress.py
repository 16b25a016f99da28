"""Decode parity on inputs that reach the online softmax's rescale paths.

With N(0,1) inputs a later key almost never beats the first tile's maximum by
the margin after which the decoders raise their reference maximum, so the
rescale of an accumulator that already holds weight would go untested.  These
inputs force it (workloads.stress_workload): logits that rise along the
sequence, dominant keys late in a sequence that many CTAs split, large |q|
(which also loads the biased-integer K products with large terms), and K/V
blocks whose scale is zero or subnormal.  Every kernel shape runs them: one
query token (head-group tiles), two to four and five tokens (one group of
consumer warps), six to eight (two groups), over the four format pairs that
matter, against the float64 oracle (TensorFold #1156, Verification: the
float64 bound holds; llama.cpp fork PR #2, the pd_combine fix: split pieces
whose maxima differ merge exactly).
"""
import os

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import assert_close, assert_lse_close, run_decode

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
F16, Q4, Q8 = W.TYPE_F16, W.TYPE_Q4_0, W.TYPE_Q8_0

# A long sequence that many CTAs split (each CTA still walks several of its
# tiles), two medium ones and a short one with a partial tile.
LENGTHS = [40000, 6000, 700, 33]
PAIRS = [(F16, F16), (Q4, Q4), (Q8, Q8), (Q8, Q4)]
NAMES = {F16: "f16", Q4: "q4_0", Q8: "q8_0"}

CASES = [(kind, kt, vt, nq) for kind in W.STRESS_KINDS for kt, vt in PAIRS for nq in (1, 3, 5, 7)]
CASES += [("rising", Q4, Q4, nq) for nq in (2, 4, 6, 8)]
CASES += [("late", Q8, Q4, nq) for nq in (2, 4, 6, 8)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_gqa_11_gb300 import _build
    _build.build()
    oracle.build()


@pytest.mark.parametrize("kind,kt,vt,nq", CASES,
                         ids=[f"{c[0]}-k{NAMES[c[1]]}-v{NAMES[c[2]]}-{c[3]}tok" for c in CASES])
def test_stress_parity(kind, kt, vt, nq):
    seed = 1000 + W.STRESS_KINDS.index(kind) * 100 + 10 * kt + vt
    w = W.stress_workload(kind, seed, LENGTHS, 16 if nq == 1 else 64, kt, vt, nq)
    go, gl = run_decode(w)
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    what = f"{kind} k{NAMES[kt]} v{NAMES[vt]} nq{nq}"
    assert_close(go, oo, what=what)
    assert_lse_close(gl, ol, what=what)
