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


@pytest.mark.parametrize("dtype,hq,hkv,d,k", [
    (torch.float16, 32, 8, 128, 3),   # two N fragments (12 columns)
    (torch.bfloat16, 16, 16, 64, 8),  # MHA, head_dim 64, 8 rows in one fragment
    (torch.bfloat16, 16, 2, 128, 2),  # GQA 8: 16 columns
    (torch.float16, 8, 1, 64, 2),     # GQA 8, head_dim 64
])
def test_short_chunks_other_shapes(dtype, hq, hkv, d, k):
    """The split-KV path for short chunks over other dtypes, head sizes and
    groups, against the C++ oracle, at lengths that end inside a 512-key
    split and exactly on one."""
    pasts = [511, 1536 - k, 1]
    B = len(pasts)
    cap = 2048
    hist = [(SI.normal((p, hkv, d), 300 + 2 * s, dtype), SI.normal((p, hkv, d), 301 + 2 * s, dtype))
            for s, p in enumerate(pasts)]
    q, kn, vn = (t.reshape(B, k, -1, d) for t in SI.gqa_prompt(B * k, seed=302, hq=hq, hkv=hkv, dim=d, dtype=dtype))
    c = Contig(dtype, hq, hkv, d, cap, batch=B, fused=True)
    for s, p in enumerate(pasts):
        c.k[s, :, :p] = hist[s][0].permute(1, 0, 2).cuda()
        c.v[s, :, :p] = hist[s][1].permute(1, 0, 2).cuda()
    c.lens.copy_(torch.tensor(pasts, dtype=torch.int32))
    out = c.chunk(q.cuda(), kn.cuda(), vn.cuda(), k, max(pasts))
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0 and c.lens.tolist() == [p + k for p in pasts]
    o = f64(out)
    worst = 0.0
    for s, p in enumerate(pasts):
        keys = np.concatenate([f64(hist[s][0]), f64(kn[s])])
        vals = np.concatenate([f64(hist[s][1]), f64(vn[s])])
        worst = max(worst, float(np.abs(o[s] - oracle.chunk_attention(f64(q[s]), keys, vals, p)).max()))
    assert worst < BF16_TOL, worst


def test_short_chunks_on_a_paged_cache():
    """4-row chunks of two sequences over 16-token pages placed by a permuted
    block table, through cp_prefill_chunk: rows against the C++ oracle, every
    new row in its page slot."""
    import chunked_prefill_causal_cp_gb300 as cp
    B, k, page = 2, 4, 16
    pasts = [1000, 37]
    need = [-(-(p + k) // page) for p in pasts]
    mb = max(need)
    perm = torch.randperm(sum(need), generator=torch.Generator().manual_seed(7)).to(torch.int32)
    table = torch.full((B, mb), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[off:off + nb]
        off += nb
    npages = sum(need)
    desc = cp.layer_desc(torch.bfloat16, B, HQ, HKV, D, cp.CP_CACHE_PAGED, page_size=page, num_pages=npages,
                         max_blocks=mb)
    kp = torch.full((npages, HKV, page, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    hist = []
    for s, p in enumerate(pasts):
        hk, hv = SI.normal((p, HKV, D), 400 + s), SI.normal((p, HKV, D), 500 + s)
        a = torch.arange(p)
        pg = table[s, a // page].long()
        kp[pg, :, a % page] = hk.cuda()
        vp[pg, :, a % page] = hv.cuda()
        hist.append((hk, hv))
    q, kn, vn = (t.reshape(B, k, -1, D) for t in SI.gqa_prompt(B * k, seed=403))
    lens = torch.tensor(pasts, dtype=torch.int32, device="cuda")
    out = torch.empty(B, k, HQ, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(cp.cp_workspace_size(desc, B * k, max(pasts) + k, B), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_prefill_chunk(desc, q.cuda(), kn.cuda(), vn.cuda(), kp, vp, lens, k, k, max(pasts), out, ws,
                        block_table=table.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and lens.tolist() == [p + k for p in pasts]
    o = f64(out)
    worst = 0.0
    for s, p in enumerate(pasts):
        a = torch.arange(p, p + k)
        pg = table[s, a // page].long()
        assert torch.equal(kp[pg, :, a % page].cpu(), kn[s]) and torch.equal(vp[pg, :, a % page].cpu(), vn[s])
        keys = np.concatenate([f64(hist[s][0]), f64(kn[s])])
        vals = np.concatenate([f64(hist[s][1]), f64(vn[s])])
        worst = max(worst, float(np.abs(o[s] - oracle.chunk_attention(f64(q[s]), keys, vals, p)).max()))
    assert worst < BF16_TOL, worst
