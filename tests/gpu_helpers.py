"""Helpers shared by the GPU parity tests: move a workload onto the device
through libpa (append kernel), run the decode, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from paged_kv_gqa_11_gb300 import PA_OK
from paged_kv_gqa_11_gb300.cache import PagedKVCache

# Attention tolerance (per element): |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL, RTOL = 2e-3, 1e-2
# Log-sum-exp tolerance (absolute, natural-log units): bounded by the largest
# logit error, which fp16 operands keep near 1e-3.
LSE_ATOL = 1e-2


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def device_cache(w: W.Workload, table=None, n_blocks=None, device="cuda"):
    """A PagedKVCache holding the workload's rows, written by the append kernel."""
    tab = w.table if table is None else table
    nb = w.n_blocks if n_blocks is None else n_blocks
    c = PagedKVCache(nb, w.page_size, w.k_type, w.v_type, device=device)
    t = to_dev(tab, device)
    if w.total_tokens:
        c.append(to_dev(w.k_rows, device), to_dev(w.v_rows, device), to_dev(w.row_seq, device),
                 to_dev(w.row_pos, device), t)
    rc = c.check()
    assert rc == PA_OK, rc
    return c, t


def run_decode(w: W.Workload, cache=None, table_dev=None, device="cuda"):
    if cache is None:
        cache, table_dev = device_cache(w, device=device)
    q = to_dev(w.q, device)
    sl = to_dev(w.seq_lens, device)
    out, lse = cache.decode(q, table_dev, sl, w.seq_lens, w.n_qtok, w.scale)
    torch.cuda.synchronize()
    rc = cache.check()
    assert rc == PA_OK, rc
    return out.cpu().numpy(), lse.cpu().numpy()


def assert_close(got: np.ndarray, want: np.ndarray, atol=ATOL, rtol=RTOL, what=""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={got[i]!r} oracle={want[i]!r} max_abs={err.max():.3g}")
    return float(err.max())


def assert_lse_close(got: np.ndarray, want: np.ndarray, what=""):
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness differs"
    if fin.any():
        d = np.abs(got[fin].astype(np.float64) - want[fin]).max()
        assert d <= LSE_ATOL, f"{what}: lse max abs err {d}"
