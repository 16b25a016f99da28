"""Writes stay inside their buffers.  Every buffer the library writes -- the
K and V pools (append), out, lse and the workspace (decode) -- is the front of
a larger allocation whose tail is poisoned; after an append and a decode at
one, three and twenty query tokens (both kernel families) every tail must come
back byte for byte, and the result must still match the oracle.  The pages ask
for bounds guards with no out-of-range access (lucebox PR #555, Validation);
a poisoned tail is the form of that check the host can read back."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, assert_lse_close, to_dev
from paged_kv_gqa_11_gb300 import PA_OK, _build
from paged_kv_gqa_11_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
TAIL = 8192
POISON = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


def _guarded(nbytes):
    """(whole allocation, view of its first nbytes); the tail holds POISON."""
    big = torch.full((nbytes + TAIL,), POISON, dtype=torch.uint8, device="cuda")
    return big, big[:nbytes]


@pytest.mark.parametrize("nq", [1, 3, 20])
def test_writes_stay_in_their_buffers(nq):
    w = W.make_workload(f"guard-{nq}", 500 + nq, [300, 64 + nq, 1000], 16, W.TYPE_Q8_0, W.TYPE_Q4_0, nq,
                        "shuffled")
    c = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type)
    k_big, c.k_pool = _guarded(c.k_pool.numel())
    v_big, c.v_pool = _guarded(c.v_pool.numel())
    c.k_pool.zero_()
    c.v_pool.zero_()
    tab = to_dev(w.table)
    c.append(to_dev(w.k_rows), to_dev(w.v_rows), to_dev(w.row_seq), to_dev(w.row_pos), tab)
    assert c.check() == PA_OK

    ws_bytes = c.workspace(w.n_seq, nq).numel()
    ws_big, c._ws = _guarded(ws_bytes)  # same size and key: decode takes this one
    n_out, n_lse = w.n_seq * nq * W.HQ * W.D * 4, w.n_seq * nq * W.HQ * 4
    out_big, out_b = _guarded(n_out)
    lse_big, lse_b = _guarded(n_lse)
    out = out_b.view(torch.float32).view(w.n_seq, nq, W.HQ, W.D)
    lse = lse_b.view(torch.float32).view(w.n_seq, nq, W.HQ)
    out, lse = c.decode(to_dev(w.q), tab, to_dev(w.seq_lens), w.seq_lens, nq, w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert c.check() == PA_OK

    for name, big, n in (("K pool", k_big, c.k_pool.numel()), ("V pool", v_big, c.v_pool.numel()),
                         ("workspace", ws_big, ws_bytes), ("out", out_big, n_out), ("lse", lse_big, n_lse)):
        tail = big[n:].cpu().numpy()
        assert (tail == POISON).all(), f"{name}: {(tail != POISON).sum()} tail bytes written"
    oo, ol = oracle.decode_workload(w, n_threads=THREADS)
    assert_close(out.cpu().numpy(), oo, what=f"guard {nq}")
    assert_lse_close(lse.cpu().numpy(), ol, what=f"guard {nq}")
