"""Checkpoint and resume: the cache and seqlens_k are the whole state of a
prompt in flight ([Wiki] 一.1-一.3).  Saving them to host memory after some
chunks, restoring them into fresh device buffers and calling the remaining
chunks gives the uninterrupted run's outputs and cache bit for bit."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, Contig, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _chunks(cache, q, k, v, sizes, start):
    outs, past = [], start
    for r in sizes:
        outs.append(cache.chunk(q[None, past:past + r], k[None, past:past + r], v[None, past:past + r], r, past)[0])
        past += r
    return outs


@pytest.mark.parametrize("fused", [True, False])
def test_resume_mid_prompt_equals_uninterrupted(fused):
    n, W = 2000, 512
    q, k, v = (t.cuda() for t in SI.gqa_prompt(n, seed=17))
    sizes = cp.cp_chunk_plan(n, W)
    whole = Contig(torch.bfloat16, 32, 8, 128, cap=2048, fused=fused)
    ref_out = torch.cat(_chunks(whole, q, k, v, sizes, 0))
    # run the first two chunks, checkpoint, and continue in fresh buffers
    first = Contig(torch.bfloat16, 32, 8, 128, cap=2048, fused=fused)
    out_a = _chunks(first, q, k, v, sizes[:2], 0)
    torch.cuda.synchronize()
    saved = (first.k.cpu(), first.v.cpu(), first.lens.cpu())
    del first
    second = Contig(torch.bfloat16, 32, 8, 128, cap=2048, fused=fused)
    second.k.copy_(saved[0])
    second.v.copy_(saved[1])
    second.lens.copy_(saved[2])
    out_b = _chunks(second, q, k, v, sizes[2:], sum(sizes[:2]))
    torch.cuda.synchronize()
    got = torch.cat(out_a + out_b)
    assert torch.equal(got, ref_out)
    assert torch.equal(second.k.view(torch.int16), whole.k.view(torch.int16))
    assert torch.equal(second.v.view(torch.int16), whole.v.view(torch.int16))
    assert int(second.lens.item()) == n and int(second.status.item()) == 0
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(got) - ref).max() < BF16_TOL
