"""GPU parity of the one-call chunk entry point (cp_prefill_chunk: append,
attention and the advance of seqlens_k in one call) against the CPU oracle and
against the same chunks run as separate append + attention calls."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, F32_TOL, Contig, f64, prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


@pytest.mark.parametrize("n,W,hq,hkv,d,dtype", [
    (700, 256, 32, 8, 128, torch.bfloat16),   # GQA 4, several tiles and a ragged tail
    (389, 128, 16, 2, 128, torch.bfloat16),   # GQA 8
    (301, 96, 4, 4, 128, torch.float16),      # MHA, chunk not a multiple of the tile
    (530, 200, 8, 2, 64, torch.bfloat16),     # head_dim 64
    (5, 2, 32, 8, 128, torch.bfloat16),       # tiny chunks, first chunk of 2 rows
])
def test_fused_chunks_match_oracle_and_separate_calls(n, W, hq, hkv, d, dtype):
    q, k, v = SI.gqa_prompt(n, seed=n, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cap = ((n + 127) // 128 + 1) * 128
    fused = Contig(dtype, hq, hkv, d, cap=cap, fused=True)
    split = Contig(dtype, hq, hkv, d, cap=cap)
    out_f, _ = prefill(fused, qd, kd, vd, W)
    out_s, _ = prefill(split, qd, kd, vd, W)
    torch.cuda.synchronize()
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(out_f) - ref).max() < BF16_TOL
    assert torch.equal(out_f, out_s)
    assert torch.equal(fused.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert torch.equal(fused.v[0, :, :n].cpu(), v.permute(1, 0, 2))
    assert int(fused.lens.item()) == n and int(fused.status.item()) == 0


def test_fused_batch_of_sequences_at_different_lengths():
    """B = 3 sequences with their own past lengths: every one is read from the
    copy of the lengths, and every one is advanced by the rows."""
    B, R, hq, hkv, d = 3, 100, 8, 2, 128
    pasts = [0, 37, 300]
    cache = Contig(torch.bfloat16, hq, hkv, d, cap=512, batch=B, fused=True)
    seqs = [SI.gqa_prompt(p + R, seed=70 + i, hq=hq, hkv=hkv, dim=d) for i, p in enumerate(pasts)]
    for b, p in enumerate(pasts):
        _, k, v = seqs[b]
        cache.k[b, :, :p] = k[:p].permute(1, 0, 2).cuda()
        cache.v[b, :, :p] = v[:p].permute(1, 0, 2).cuda()
    cache.lens.copy_(torch.tensor(pasts, dtype=torch.int32))
    qb = torch.stack([s[0][p:p + R] for s, p in zip(seqs, pasts)]).cuda()
    kb = torch.stack([s[1][p:p + R] for s, p in zip(seqs, pasts)]).cuda()
    vb = torch.stack([s[2][p:p + R] for s, p in zip(seqs, pasts)]).cuda()
    out = cache.chunk(qb, kb, vb, R, max(pasts))
    torch.cuda.synchronize()
    for b, p in enumerate(pasts):
        q, k, v = seqs[b]
        ref = oracle.chunk_attention(f64(q[p:p + R]), f64(k), f64(v), p)
        assert np.abs(f64(out[b]) - ref).max() < BF16_TOL
        assert torch.equal(cache.k[b, :, p:p + R].cpu(), k[p:p + R].permute(1, 0, 2))
    assert cache.lens.tolist() == [p + R for p in pasts]


def test_fused_padding_ladder_equals_separate_calls():
    """A widened last chunk: the real rows and the cache are bit-identical to
    the separate calls, and seqlens_k advances by the real rows only."""
    idx = 1
    n = SI.LADDER_PROMPT_LENGTHS[idx]
    q, k, v = SI.ladder_prompt(idx)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fused = Contig(torch.bfloat16, 32, 8, 128, cap=8192, fused=True)
    split = Contig(torch.bfloat16, 32, 8, 128, cap=8192)
    out_f, widths = prefill(fused, qd, kd, vd, 512, pad=True)
    out_s, _ = prefill(split, qd, kd, vd, 512, pad=True)
    torch.cuda.synchronize()
    assert widths[-1] > n - 512 * (len(widths) - 1)  # the last chunk was widened
    assert torch.equal(out_f, out_s)
    assert torch.equal(fused.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert int(fused.lens.item()) == n and int(fused.status.item()) == 0


@pytest.mark.parametrize("n,hq,hkv,d,dtype", [
    (3000, 32, 8, 128, torch.bfloat16),  # split-KV decode path, then a separate advance
    (1, 32, 8, 128, torch.bfloat16),     # first token
    (700, 8, 4, 64, torch.float16),      # GQA 2, head_dim 64
])
def test_fused_decode_row(n, hq, hkv, d, dtype):
    q, k, v = SI.gqa_prompt(n, seed=9 + n, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    cache = Contig(dtype, hq, hkv, d, cap=((n + 127) // 128 + 1) * 128, fused=True)
    cache.k[0, :, :n - 1] = k[:n - 1].permute(1, 0, 2).cuda()
    cache.v[0, :, :n - 1] = v[:n - 1].permute(1, 0, 2).cuda()
    cache.lens.fill_(n - 1)
    out = cache.chunk(q[None, n - 1:].cuda(), k[None, n - 1:].cuda(), v[None, n - 1:].cuda(), 1, n - 1)
    torch.cuda.synchronize()
    ref = oracle.attention_row(f64(q[n - 1]), f64(k), f64(v), n - 1)
    assert np.abs(f64(out[0, 0]) - ref).max() < BF16_TOL
    assert torch.equal(cache.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert int(cache.lens.item()) == n and int(cache.status.item()) == 0


def test_fused_fp32_glossary_example():
    """fp32 (the SIMT path, one launch per chunk): 1e-4 of the oracle."""
    q, k, v = SI.fp32_sdpa_example()
    cache = Contig(torch.float32, 8, 8, 64, cap=1024, fused=True)
    out, _ = prefill(cache, q.cuda(), k.cuda(), v.cuda(), 256)
    torch.cuda.synchronize()
    ref = oracle.causal_attention(f64(q), f64(k), f64(v))
    assert np.abs(f64(out) - ref).max() < F32_TOL
    assert int(cache.lens.item()) == 1000 and int(cache.status.item()) == 0


@pytest.mark.parametrize("n,W,hq,hkv,d", [
    (700, 256, 8, 2, 64),    # GQA 4, head_dim 64 (four warp groups split the keys)
    (389, 128, 4, 2, 128),   # GQA 2, head_dim 128 (two warp groups)
    (301, 96, 4, 4, 64),     # MHA, chunk not a multiple of the 32-key tile
    (5, 2, 8, 4, 128),       # tiny chunks, first chunk of 2 rows
])
def test_fused_fp32_chunks_match_oracle_and_separate_calls(n, W, hq, hkv, d):
    """fp32 on a contiguous cache is one launch per chunk (the kernel reads the
    chunk's keys from k_new, copies its rows into the cache and advances
    seqlens_k by ticket): within 1e-4 of the oracle, bit-identical to the
    separate append + attention calls, and the cache byte for byte."""
    q, k, v = SI.gqa_prompt(n, seed=n + 1, hq=hq, hkv=hkv, dim=d, dtype=torch.float32)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cap = ((n + 127) // 128 + 1) * 128
    fused = Contig(torch.float32, hq, hkv, d, cap=cap, fused=True)
    split = Contig(torch.float32, hq, hkv, d, cap=cap)
    out_f, _ = prefill(fused, qd, kd, vd, W)
    out_s, _ = prefill(split, qd, kd, vd, W)
    torch.cuda.synchronize()
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(out_f) - ref).max() < F32_TOL
    assert torch.equal(out_f, out_s)
    assert torch.equal(fused.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert torch.equal(fused.v[0, :, :n].cpu(), v.permute(1, 0, 2))
    assert torch.isnan(fused.k[0, :, n:]).all()
    assert int(fused.lens.item()) == n and int(fused.status.item()) == 0
    assert int(fused.ws[:4].view(torch.int32).item()) == 0  # the ticket counter is left zero


def test_fused_fp32_batch_padded_chunk():
    """fp32, B = 3 sequences at their own lengths, one chunk widened from 90 to
    100 rows (the pad rows repeat the last real row): every sequence's real rows
    within 1e-4 of the oracle, its 100 rows appended, each length advanced by
    the 90 real rows."""
    B, R, real, hq, hkv, d = 3, 100, 90, 8, 2, 64
    pasts = [0, 37, 300]
    cache = Contig(torch.float32, hq, hkv, d, cap=512, batch=B, fused=True)
    seqs = [SI.gqa_prompt(p + real, seed=80 + i, hq=hq, hkv=hkv, dim=d, dtype=torch.float32)
            for i, p in enumerate(pasts)]
    for b, p in enumerate(pasts):
        _, k, v = seqs[b]
        cache.k[b, :, :p] = k[:p].permute(1, 0, 2).cuda()
        cache.v[b, :, :p] = v[:p].permute(1, 0, 2).cuda()
    cache.lens.copy_(torch.tensor(pasts, dtype=torch.int32))

    def widened(t, p):
        idx = torch.cat([torch.arange(p, p + real), torch.full((R - real,), p + real - 1)])
        return t[idx]

    qb = torch.stack([widened(s[0], p) for s, p in zip(seqs, pasts)]).cuda()
    kb = torch.stack([widened(s[1], p) for s, p in zip(seqs, pasts)]).cuda()
    vb = torch.stack([widened(s[2], p) for s, p in zip(seqs, pasts)]).cuda()
    out = cache.chunk(qb, kb, vb, real, max(pasts))
    torch.cuda.synchronize()
    for b, p in enumerate(pasts):
        q, k, v = seqs[b]
        ref = oracle.chunk_attention(f64(q[p:p + real]), f64(k), f64(v), p)
        assert np.abs(f64(out[b, :real]) - ref).max() < F32_TOL
        assert torch.equal(cache.k[b, :, p:p + R].cpu(), kb[b].cpu().permute(1, 0, 2))
        assert torch.equal(cache.v[b, :, p:p + R].cpu(), vb[b].cpu().permute(1, 0, 2))
    assert cache.lens.tolist() == [p + real for p in pasts]
    assert int(cache.status.item()) == 0


def test_fused_paged_prompt():
    """A prompt over a paged pool with permuted pages (the tensor-core kernel
    reads this call's own tiles from k_new / v_new)."""
    n, W, hq, hkv, d, ps = 900, 256, 16, 4, 128, 32
    q, k, v = SI.gqa_prompt(n, seed=5, hq=hq, hkv=hkv, dim=d)
    nb = (n + ps - 1) // ps + 1
    perm = torch.randperm(nb * 2, generator=torch.Generator().manual_seed(5))[:nb].to(torch.int32)
    desc = cp.layer_desc(torch.bfloat16, 1, hq, hkv, d, cp.CP_CACHE_PAGED, page_size=ps, num_pages=nb * 2,
                         max_blocks=nb)
    kp = torch.full((nb * 2, hkv, ps, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    table = perm[None].cuda()
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(cp.cp_workspace_size(desc, W, nb * ps, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty(n, hq, d, dtype=torch.bfloat16, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    past = 0
    for r in cp.cp_chunk_plan(n, W):
        sl = slice(past, past + r)
        cp.cp_prefill_chunk(desc, qd[None, sl].contiguous(), kd[None, sl].contiguous(), vd[None, sl].contiguous(),
                            kp, vp, lens, r, r, past, out[None, sl], ws, block_table=table, dev_status=status)
        past += r
    torch.cuda.synchronize()
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(out) - ref).max() < BF16_TOL
    assert int(lens.item()) == n and int(status.item()) == 0
    a = torch.arange(n)
    pages = perm[(a // ps).long()].long()
    assert torch.equal(kp[pages, :, a % ps].cpu(), k)
