"""GPU parity of short chunks at long cached lengths: a k-row chunk (k = 2..8,
a speculative-verify step in the glossary's related techniques, or a prefix
cache hit resuming at past > 0) for several sequences at different lengths,
up to the cache's capacity, through the one-call and the separate-call
entry points: rows against the C++ oracle, the two paths bit-identical, the
cache byte for byte."""
import numpy as np
import pytest
import torch

import synth_inputs as SI
from gpu_util import BF16_TOL, Contig, f64
from oracle import cpp as oracle

pytestmark = pytest.mark.gpu

HQ, HKV, D, CAP = 32, 8, 128, 8192


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


@pytest.mark.parametrize("k", [2, 3, 5, 8])
def test_k_row_chunk_at_long_past(k):
    pasts = [4000, CAP - k, 37]
    B = len(pasts)
    hist = [(SI.normal((p, HKV, D), 90 + 2 * s), SI.normal((p, HKV, D), 91 + 2 * s)) for s, p in enumerate(pasts)]
    q, kn, vn = (t.reshape(B, k, -1, D) for t in SI.gqa_prompt(B * k, seed=92 + k))
    outs = []
    caches = []
    for fused in (True, False):
        c = Contig(torch.bfloat16, HQ, HKV, D, CAP, batch=B, fused=fused)
        for s, p in enumerate(pasts):
            c.k[s, :, :p] = hist[s][0].permute(1, 0, 2).cuda()
            c.v[s, :, :p] = hist[s][1].permute(1, 0, 2).cuda()
        c.lens.copy_(torch.tensor(pasts, dtype=torch.int32))
        outs.append(c.chunk(q.cuda(), kn.cuda(), vn.cuda(), k, max(pasts)))
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0
        assert c.lens.tolist() == [p + k for p in pasts]
        caches.append(c)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0].k.view(torch.int16), caches[1].k.view(torch.int16))
    assert torch.equal(caches[0].v.view(torch.int16), caches[1].v.view(torch.int16))
    o = f64(outs[0])
    worst = 0.0
    for s, p in enumerate(pasts):
        got = caches[0].k[s].permute(1, 0, 2)
        assert torch.equal(got[p:p + k].cpu(), kn[s]) and torch.equal(caches[0].v[s].permute(1, 0, 2)[p:p + k].cpu(), vn[s])
        assert torch.isnan(got[p + k:].float()).all()
        keys = np.concatenate([f64(hist[s][0]), f64(kn[s])])
        vals = np.concatenate([f64(hist[s][1]), f64(vn[s])])
        ref = oracle.chunk_attention(f64(q[s]), keys, vals, p)
        worst = max(worst, float(np.abs(o[s] - ref).max()))
    assert worst < BF16_TOL, worst
