"""Failure detection on the GPU without a fault: the bounded wait that every
kernel of the library uses gives up on a barrier that nothing completes,
reports CP_DEV_TIMEOUT through the status word, and leaves the context usable
(a chunk call right after it is checked against the oracle)."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, Contig, f64, prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(5, dtype=torch.int64, device="cuda")
    assert cp.cp_selftest_bounded_wait(status, out) == cp.CP_OK
    torch.cuda.synchronize()  # raises if the context was lost
    ok1, t1, ok2, t2, aborted = out.tolist()
    assert int(status.item()) == cp.CP_DEV_TIMEOUT
    assert ok1 == 0 and ok2 == 0 and aborted == 1
    assert 4.0e9 <= t1 < 6.0e9, t1   # the first wait ran to the 4 s limit
    assert t2 < 1.0e8, t2            # the second returned at once (the CTA had aborted)
    # The same process and context still run the library's kernels correctly.
    n, W = 300, 128
    q, k, v = SI.gqa_prompt(n, seed=9)
    cache = Contig(torch.bfloat16, 32, 8, 128, cap=384, fused=True)
    o, _ = prefill(cache, q.cuda(), k.cuda(), v.cuda(), W)
    torch.cuda.synchronize()
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(o) - ref).max() < BF16_TOL
    assert int(cache.status.item()) == 0
