"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code running under a device-memory
budget fixed at start-up, hot loops that must not take cudaMalloc's implicit
device synchronisation, plain C code with no allocator.  For them the library
offers one entry point whose scratch is a fixed static device array instead of
a caller workspace.  These tests call it through the C ABI and check it
against the workspace entry point (pa_decode) on two calls in a row, and that
a batch too large for the array is refused.  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import ATOL, RTOL, assert_close, device_cache, to_dev
import paged_kv_gqa_11_gb300 as pa
from paged_kv_gqa_11_gb300 import _build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


CASES = [
    # one query token (head-group tiles), the ragged long-context shape
    ("q4-1tok", [20000, 513, 3000, 64], 16, W.TYPE_Q4_0, 1),
    # four query tokens (per-head tiles), verify-width shape
    ("q8-4tok", [9000, 777, 130], 256, W.TYPE_Q8_0, 4),
]


@pytest.mark.parametrize("name,lens,ps,kt,nq", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point(name, lens, ps, kt, nq):
    w = W.make_workload(name, 31, lens, ps, kt, kt, nq, "shuffled")
    cache, table = device_cache(w)
    q = to_dev(w.q)
    sl_dev = to_dev(w.seq_lens)
    sl_host = np.ascontiguousarray(w.seq_lens, np.int32)
    ref_out, ref_lse = cache.decode(q, table, sl_dev, sl_host, nq, w.scale)
    torch.cuda.synchronize()
    assert cache.check() == pa.PA_OK
    ref_out, ref_lse = ref_out.cpu().numpy(), ref_lse.cpu().numpy()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.n_seq, nq, W.HQ), float("nan"), device=q.device)
        rc = pa.pa_decode_noalloc(cache.pool, q, cache.k_pool, cache.v_pool, table, table.shape[1], sl_dev, sl_host,
                                  w.n_seq, nq, W.HQ, w.scale, out, lse, cache.err)
        assert rc == pa.PA_OK, pa.status_name(rc)
        torch.cuda.synchronize()
        assert cache.check() == pa.PA_OK
        assert_close(out.cpu().numpy(), ref_out.astype(np.float64), ATOL, RTOL, what=f"{name} call {call}")
        got_lse = lse.cpu().numpy()
        assert np.allclose(got_lse, ref_lse, rtol=RTOL, atol=ATOL), f"{name} call {call}: lse"


def test_noalloc_refuses_batches_beyond_the_scratch():
    p = pa.Pool(64, 16, 4, 256, pa.PA_Q4_0)
    dev = torch.cuda.current_device()
    n_seq = 100000
    assert pa.pa_decode_workspace_size(p, n_seq, 1, dev) > pa.NOALLOC_SCRATCH_BYTES
    sl = np.full(n_seq, 16, np.int32)
    # rejected on the host before any launch (the pointers are never used)
    rc = pa.pa_decode_noalloc(p, 4096, 4096, 4096, 4096, 1, 4096, sl, n_seq, 1, 24, 0.0625, 4096, None, 4096,
                              stream=None)
    assert rc == pa.PA_ERR_UNSUPPORTED
