"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code running under a device-memory
budget fixed at start-up, hot loops that must not take cudaMalloc's implicit
device synchronisation, plain C code with no allocator.  For them the library
offers one entry point whose scratch is a fixed static device array instead of
a caller workspace.  These tests call it through the C ABI and check that its
results are bit-identical to the workspace entry point's (pa_decode runs the
same kernels with the same plan), over calls in a row whose shapes differ, so
that anything a call left in the shared array would show in the next; and that
a batch too large for the array is refused.  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import device_cache, to_dev
import paged_kv_gqa_11_gb300 as pa
from paged_kv_gqa_11_gb300 import _build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


CASES = {
    # one query token (head-group tiles), the ragged long-context shape
    "q4-1tok": ([20000, 513, 3000, 64], 16, W.TYPE_Q4_0, 1),
    # four query tokens (per-head tiles), a verify-width shape
    "q8-4tok": ([9000, 777, 130], 256, W.TYPE_Q8_0, 4),
    # more sequences than one launch takes: sub-batches through the one array
    "q8-3tok-300seq": ([40 + (37 * i) % 500 for i in range(300)], 16, W.TYPE_Q8_0, 3),
    # row tiles (tcgen05 kernel), two row tiles per KV head, a sequence with L = n_qtok
    "q8-40tok": ([3000, 40, 700], 16, W.TYPE_Q8_0, 40),
}


def _both(name):
    lens, ps, kt, nq = CASES[name]
    w = W.make_workload(name, 31, lens, ps, kt, kt, nq, "shuffled")
    cache, table = device_cache(w)
    q = to_dev(w.q)
    sl_dev = to_dev(w.seq_lens)
    sl_host = np.ascontiguousarray(w.seq_lens, np.int32)
    ref_out, ref_lse = cache.decode(q, table, sl_dev, sl_host, nq, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == pa.PA_OK
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_seq, nq, W.HQ), float("nan"), device=q.device)
    rc = pa.pa_decode_noalloc(cache.pool, q, cache.k_pool, cache.v_pool, table, table.shape[1], sl_dev, sl_host,
                              w.n_seq, nq, W.HQ, w.scale, out, lse, cache.err)
    assert rc == pa.PA_OK, pa.status_name(rc)
    torch.cuda.synchronize()
    assert cache.check() == pa.PA_OK
    return (ref_out.cpu().numpy(), ref_lse.cpu().numpy()), (out.cpu().numpy(), lse.cpu().numpy())


def test_noalloc_is_bit_identical_over_calls_of_different_shapes():
    for call, name in enumerate(["q4-1tok", "q8-4tok", "q8-40tok", "q8-3tok-300seq", "q4-1tok", "q8-40tok"]):
        (ro, rl), (go, gl) = _both(name)
        assert np.isfinite(go).all(), f"call {call} ({name})"
        assert np.array_equal(go, ro), f"call {call} ({name}): out differs from pa_decode"
        assert np.array_equal(gl, rl), f"call {call} ({name}): lse differs from pa_decode"


def test_noalloc_refuses_batches_beyond_the_scratch():
    """A call whose scratch would exceed the array is refused on the host,
    before any launch (the pointers are never used).  One launch takes at most
    128 sequences, so the scratch a call needs is bounded; the row tiles' 128
    partial rows per segment take it past the array at 96 query tokens."""
    p = pa.Pool(64, 16, 4, 256, pa.PA_Q4_0)
    dev = torch.cuda.current_device()
    n_seq = 100000
    refused = 0
    for nq in list(range(1, 9)) + [20, 96]:  # decode kernels and row tiles
        sl = np.full(n_seq, max(16, nq), np.int32)
        need = pa.pa_decode_workspace_size(p, n_seq, nq, dev)
        assert need > 0
        if need > pa.NOALLOC_SCRATCH_BYTES:
            rc = pa.pa_decode_noalloc(p, 4096, 4096, 4096, 4096, 1, 4096, sl, n_seq, nq, 24, 0.0625, 4096, None,
                                      4096, stream=None)
            assert rc == pa.PA_ERR_UNSUPPORTED
            refused += 1
    if refused == 0:
        pytest.skip("every shape's scratch fits the array on this device")
