"""GPU parity of the contiguous-cache path (append + chunk attention + commit)
against the CPU oracle, through the C ABI."""
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


def test_fp32_glossary_example_chunked_equals_one_shot():
    """1000 tokens, chunks 256/256/256/232, 8 heads x 64, fp32: the GPU chunked
    output matches the oracle's one-shot causal attention within 1e-4, and the
    cache after each chunk is the prefix of the one-shot cache, bit for bit."""
    q, k, v = SI.fp32_sdpa_example()
    cache = Contig(torch.float32, 8, 8, 64, cap=1024)
    out, widths = prefill(cache, q.cuda(), k.cuda(), v.cuda(), 256)
    torch.cuda.synchronize()
    assert widths == [256, 256, 256, 232]
    ref = oracle.causal_attention(f64(q), f64(k), f64(v))
    err = np.abs(f64(out) - ref).max()
    assert err < F32_TOL, err
    assert torch.equal(cache.k[0, :, :1000].cpu(), k.permute(1, 0, 2))
    assert torch.isnan(cache.k[0, :, 1000:]).all()
    assert int(cache.lens.item()) == 1000 and int(cache.status.item()) == 0


@pytest.mark.parametrize("n,W,hq,hkv,d,dtype", [
    (700, 256, 32, 8, 128, torch.bfloat16),   # GQA 4, several tiles and a ragged tail
    (389, 128, 16, 2, 128, torch.bfloat16),   # GQA 8
    (301, 96, 4, 4, 128, torch.float16),      # MHA, chunk not a multiple of the tile
    (530, 200, 8, 2, 64, torch.bfloat16),     # head_dim 64
    (257, 257, 16, 1, 64, torch.float16),     # GQA 16, one chunk
    (5, 2, 32, 8, 128, torch.bfloat16),       # tiny chunks, first chunk of 2 rows
])
def test_chunked_prefill_elementwise(n, W, hq, hkv, d, dtype):
    q, k, v = SI.gqa_prompt(n, seed=n, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    cache = Contig(dtype, hq, hkv, d, cap=((n + 127) // 128 + 1) * 128)
    out, _ = prefill(cache, q.cuda(), k.cuda(), v.cuda(), W)
    torch.cuda.synchronize()
    ref, snaps, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    err = np.abs(f64(out) - ref).max()
    assert err < BF16_TOL, err
    assert np.isfinite(f64(out)).all()
    assert torch.equal(cache.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert torch.equal(cache.v[0, :, :n].cpu(), v.permute(1, 0, 2))
    assert int(cache.status.item()) == 0


def test_gqa_prompt_4000_full_size():
    """The GQA 32/8 x 128 bf16 prompt of 4000 tokens in chunks of 512 (7x512+416)
    over a cache of physical capacity 8192 poisoned with NaN past the valid
    length: every chunk's first/last rows and 24 seeded rows per chunk match
    the oracle one by one; the cache after each chunk equals the prefix of the
    prompt's K/V byte for byte and the rest stays untouched."""
    n, W = 4000, 512
    q, k, v = SI.gqa_prompt(n, seed=1)
    cache = Contig(torch.bfloat16, 32, 8, 128, cap=8192)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    past = 0
    sizes = cp.cp_chunk_plan(n, W)
    assert sizes == [512] * 7 + [416]
    for r in sizes:
        out[past:past + r] = cache.chunk(qd[None, past:past + r], kd[None, past:past + r],
                                         vd[None, past:past + r], r, past)[0]
        past += r
        assert torch.equal(cache.k[0, :, :past].cpu(), k[:past].permute(1, 0, 2))
        assert torch.isnan(cache.k[0, :, past:].float()).all()
    torch.cuda.synchronize()
    assert int(cache.lens.item()) == n and int(cache.status.item()) == 0
    rng = np.random.default_rng(0)
    rows = []
    start = 0
    for r in sizes:
        rows += [start, start + r - 1] + list(rng.integers(start, start + r, 24))
        start += r
    kk, vv, qq, oo = f64(k), f64(v), f64(q), f64(out)
    worst = 0.0
    for p in rows:
        ref = oracle.attention_row(qq[p], kk, vv, int(p))
        worst = max(worst, np.abs(oo[p] - ref).max())
    assert worst < BF16_TOL, worst
    assert np.isfinite(oo).all()


def test_batch_of_sequences_at_different_lengths():
    """B = 3 sequences in one call, each with its own past length."""
    B, R, hq, hkv, d = 3, 100, 8, 2, 128
    pasts = [0, 37, 300]
    cap = 512
    cache = Contig(torch.bfloat16, hq, hkv, d, cap=cap, batch=B)
    seqs = [SI.gqa_prompt(p + R, seed=70 + i, hq=hq, hkv=hkv, dim=d) for i, p in enumerate(pasts)]
    for b, p in enumerate(pasts):  # pre-fill each past
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
    assert cache.lens.tolist() == [p + R for p in pasts]


@pytest.mark.parametrize("idx", range(len(SI.LADDER_PROMPT_LENGTHS)))
def test_query_padding_ladder(idx):
    """Query-axis padding: each prompt's chunks are widened to {171,342,512} by
    repeating the last real row; real rows are bit-identical to the unpadded
    run, a second run of the same prompt is bit-identical too, the cache is
    rewound to past + real rows after each chunk (pad K/V sit beyond it until
    the next chunk overwrites them), and the rows match the oracle."""
    n = SI.LADDER_PROMPT_LENGTHS[idx]
    q, k, v = SI.ladder_prompt(idx)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    plain = Contig(torch.bfloat16, 32, 8, 128, cap=8192)
    ref_out, w0 = prefill(plain, qd, kd, vd, 512, pad=False)
    outs, caches = [], []
    for _ in range(2):  # each prompt is run twice
        padded = Contig(torch.bfloat16, 32, 8, 128, cap=8192)
        o, widths = prefill(padded, qd, kd, vd, 512, pad=True)
        outs.append(o)
        caches.append(padded)
    torch.cuda.synchronize()
    assert set(widths) <= {171, 342, 512}
    assert widths[-1] == cp.cp_query_width(n - 512 * (len(widths) - 1), 512)
    assert torch.equal(outs[0], ref_out) and torch.equal(outs[1], ref_out)
    for c in caches:
        assert int(c.lens.item()) == n and int(c.status.item()) == 0
        assert torch.equal(c.k[0, :, :n].cpu(), k.permute(1, 0, 2))
        # pad slots of the last chunk hold copies of the last real row
        extra = widths[-1] - (n - 512 * (len(widths) - 1))
        if extra:
            tail = c.k[0, :, n:n + extra].cpu()
            assert torch.equal(tail, k[n - 1].unsqueeze(1).expand_as(tail))
    rng = np.random.default_rng(idx)
    kk, vv, qq, oo = f64(k), f64(v), f64(q), f64(ref_out)
    for p in [0, n - 1] + list(rng.integers(0, n, 16)):
        assert np.abs(oo[p] - oracle.attention_row(qq[p], kk, vv, int(p))).max() < BF16_TOL


@pytest.mark.parametrize("n,hq,hkv,d,dtype", [
    (3000, 32, 8, 128, torch.bfloat16),  # GQA 4, several 512-key splits and a ragged last one
    (1, 32, 8, 128, torch.bfloat16),     # first token: the row sees only itself
    (1537, 16, 2, 128, torch.bfloat16),  # GQA 8, one key past a split boundary
    (700, 8, 4, 64, torch.float16),      # GQA 2, head_dim 64
    (512, 8, 8, 64, torch.float16),      # MHA, exactly one split
    (900, 16, 1, 64, torch.bfloat16),    # GQA 16 (goes to the tensor-core kernel)
])
def test_decode_row_through_prefill_call(n, hq, hkv, d, dtype):
    """A one-row chunk (a decode step) over a contiguous context takes the
    split-KV path (the tensor-core path for groups wider than 8) and matches
    the oracle."""
    q, k, v = SI.gqa_prompt(n, seed=9 + n, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    cache = Contig(dtype, hq, hkv, d, cap=((n + 127) // 128 + 1) * 128)
    cache.k[0, :, :n - 1] = k[:n - 1].permute(1, 0, 2).cuda()
    cache.v[0, :, :n - 1] = v[:n - 1].permute(1, 0, 2).cuda()
    cache.lens.fill_(n - 1)
    out = cache.chunk(q[None, n - 1:].cuda(), k[None, n - 1:].cuda(), v[None, n - 1:].cuda(), 1, n - 1)
    torch.cuda.synchronize()
    ref = oracle.attention_row(f64(q[n - 1]), f64(k), f64(v), n - 1)
    assert np.abs(f64(out[0, 0]) - ref).max() < BF16_TOL
    assert torch.equal(cache.k[0, :, :n].cpu(), k.permute(1, 0, 2))
    assert int(cache.status.item()) == 0


def test_out_of_range_length_is_reported_not_read():
    """A seqlens_k value beyond the host bound is skipped and reported in the
    device status word instead of being used to address the cache."""
    cache = Contig(torch.bfloat16, 8, 2, 128, cap=256)
    q, k, v = SI.gqa_prompt(64, seed=3, hq=8, hkv=2)
    cache.lens.fill_(250)  # 250 + 64 > 256, but the host was told max_past = 0
    out = torch.zeros(1, 64, 8, 128, dtype=torch.bfloat16, device="cuda")
    cp.cp_kv_append(cache.desc, k[None].cuda(), v[None].cuda(), 64, cache.k, cache.v, cache.lens, 0,
                    dev_status=cache.status)
    cp.cp_prefill_chunk_attn(cache.desc, q[None].cuda(), cache.k, cache.v, cache.lens, 64, 64, 0, out,
                             cache.ws, commit=False, dev_status=cache.status)
    torch.cuda.synchronize()
    assert int(cache.status.item()) & cp.CP_DEV_BOUNDS
    assert torch.isnan(cache.k.float()).all()  # nothing was written
