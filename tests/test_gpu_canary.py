"""Canary bands around every buffer an entry point writes, checked bit for bit
after the call, and the read-only inputs checked unchanged: no launch writes
outside its output rows or into its inputs.  Each case also checks its
output against the oracle, so the bands guard a result that is right."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, F32_TOL, f64

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side (8 or 16 KB: keeps the view 16-byte aligned)
SENTINEL = {2: 0x7F5A, 4: 0x7FC5A5A5}  # NaN bit patterns with a payload no kernel writes


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def guarded(shape, dtype, fill=None):
    """(buffer, view): `view` of `shape` inside a buffer whose GUARD elements on
    each side hold the sentinel; the view itself holds `fill` (or the sentinel)."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    _bits(buf).fill_(SENTINEL[buf.element_size()])
    view = buf[GUARD:GUARD + n].view(shape)
    if fill is not None:
        view.copy_(fill)
    return buf, view


def bands_intact(buf):
    s = SENTINEL[buf.element_size()]
    b = _bits(buf)
    return bool((b[:GUARD] == s).all()) and bool((b[-GUARD:] == s).all())


def test_contiguous_chunks_stay_in_their_rows():
    """One-call chunks on a contiguous cache (bf16 tensor-core launch, then a
    decode row on the split-KV path): output, cache and workspace bands
    intact, q/k/v unchanged, slots past the length still NaN."""
    n, W, hq, hkv, d, cap = 530, 256, 32, 8, 128, 640
    q, k, v = SI.gqa_prompt(n + 1, seed=3, hq=hq, hkv=hkv, dim=d)
    desc = cp.layer_desc(torch.bfloat16, 1, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=cap)
    kb, kc = guarded((1, hkv, cap, d), torch.bfloat16, float("nan"))
    vb, vc = guarded((1, hkv, cap, d), torch.bfloat16, float("nan"))
    wsz = cp.cp_workspace_size(desc, 16, cap, 1)
    wb, ws16 = guarded(((wsz + 1) // 2,), torch.int16, 0)  # zeroed, in 2-byte elements for the sentinel
    ws = ws16.view(torch.uint8)
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    past = 0
    for r in cp.cp_chunk_plan(n, W) + [1]:
        qd, kd, vd = (t[past:past + r][None].cuda() for t in (q, k, v))
        keep = [t.clone() for t in (qd, kd, vd)]
        ob, out = guarded((1, r, hq, d), torch.bfloat16)
        cp.cp_prefill_chunk(desc, qd, kd, vd, kc, vc, lens, r, r, past, out, ws, dev_status=status)
        torch.cuda.synchronize()
        assert bands_intact(ob), (past, r)
        assert all(torch.equal(_bits(a), _bits(b)) for a, b in zip(keep, (qd, kd, vd)))
        outs.append(out[0].clone())
        past += r
    assert int(status.item()) == 0 and int(lens.item()) == n + 1
    assert bands_intact(kb) and bands_intact(vb) and bands_intact(wb)
    assert torch.isnan(kc[0, :, n + 1:].float()).all() and torch.isnan(vc[0, :, n + 1:].float()).all()
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)  # the decode row is one more chunk of 1
    got = f64(torch.cat(outs))
    assert np.abs(got[:n] - ref[:n]).max() < BF16_TOL
    row = oracle.attention_row(f64(q)[n], f64(k), f64(v), n)
    assert np.abs(got[n] - row).max() < BF16_TOL


def test_fp32_chunk_stays_in_its_rows():
    """The fp32 one-launch chunk: output and cache bands intact, inputs unchanged."""
    n, W, h, d, cap = 300, 128, 8, 64, 300
    q, k, v = SI.gqa_prompt(n, seed=4, hq=h, hkv=h, dim=d, dtype=torch.float32)
    desc = cp.layer_desc(torch.float32, 1, h, h, d, cp.CP_CACHE_CONTIG, capacity=cap)
    kb, kc = guarded((1, h, cap, d), torch.float32, float("nan"))
    vb, vc = guarded((1, h, cap, d), torch.float32, float("nan"))
    ws = torch.zeros(cp.cp_workspace_size(desc, W, cap, 1), dtype=torch.uint8, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ob, out = guarded((1, n, h, d), torch.float32)
    past = 0
    for r in cp.cp_chunk_plan(n, W):
        qd, kd, vd = (t[past:past + r][None].cuda() for t in (q, k, v))
        keep = [t.clone() for t in (qd, kd, vd)]
        o = out[:, past:past + r]
        cp.cp_prefill_chunk(desc, qd, kd, vd, kc, vc, lens, r, r, past, o, ws, dev_status=status)
        torch.cuda.synchronize()
        assert all(torch.equal(_bits(a), _bits(b)) for a, b in zip(keep, (qd, kd, vd)))
        past += r
    assert int(status.item()) == 0 and bands_intact(ob) and bands_intact(kb) and bands_intact(vb)
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(out[0]) - ref).max() < F32_TOL


def test_ring_chunks_stay_in_their_rows():
    """One-call chunks on a ring (the ring instantiation): output and ring bands intact."""
    n_real, c, C, h, d = 500, 96, 352, 4, 128
    L = cp.cp_aligned_length(n_real, c)
    q, k, v = SI.rolling_prompt(L, seed=6, heads=h, dim=d, dtype=torch.float16)
    desc = cp.layer_desc(torch.float16, 1, h, h, d, cp.CP_CACHE_ROLLING, capacity=C)
    kb, kc = guarded((1, h, C, d), torch.float16, float("nan"))
    vb, vc = guarded((1, h, C, d), torch.float16, float("nan"))
    ws = torch.zeros(cp.cp_workspace_size(desc, c, C, 1), dtype=torch.uint8, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    left = torch.tensor([L - n_real], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ob, out = guarded((1, L, h, d), torch.float16)
    for ci in range(L // c):
        sl = slice(ci * c, (ci + 1) * c)
        qd, kd, vd = (t[sl][None].contiguous().cuda() for t in (q, k, v))
        cp.cp_prefill_chunk(desc, qd, kd, vd, kc, vc, lens, c, c, ci * c, out[:, sl], ws, left_pad=left,
                            dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bands_intact(ob) and bands_intact(kb) and bands_intact(vb)
    ref, _ = oracle.rolling_prefill(f64(q), f64(k), f64(v), c, C, L - n_real)
    assert np.abs(f64(out[0])[L - n_real:] - ref[L - n_real:]).max() < BF16_TOL


def test_mixed_step_stays_in_its_rows():
    """A paged mixed step (two decode rows and a prompt chunk over cached
    pages): output, pool and table bands intact, inputs unchanged, unused pages NaN."""
    page, hq, hkv, d = 16, 32, 8, 128
    hist = [300, 1029, 700]
    rows = [1, 1, 200]
    need = [-(-(p + r) // page) for p, r in zip(hist, rows)]
    max_blocks, num_pages = max(need), sum(need) + 3  # three pages no sequence uses
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(2))
    table = torch.full((3, max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    desc = cp.layer_desc(torch.bfloat16, 0, hq, hkv, d, cp.CP_CACHE_PAGED, page_size=page, num_pages=num_pages,
                         max_blocks=max_blocks)
    kb, kp = guarded((num_pages, hkv, page, d), torch.bfloat16, float("nan"))
    vb, vp = guarded((num_pages, hkv, page, d), torch.bfloat16, float("nan"))
    ok = np.full(tuple(kp.shape), np.nan)
    ov = np.full(tuple(kp.shape), np.nan)
    for s, n in enumerate(hist):
        hk, hv = SI.normal((n, hkv, d), 60 + s).bfloat16(), SI.normal((n, hkv, d), 70 + s).bfloat16()
        a = torch.arange(n)
        pg = table[s, a // page].long()
        kp[pg, :, a % page] = hk.cuda()
        vp[pg, :, a % page] = hv.cuda()
        ok[pg.numpy(), :, (a % page).numpy()] = f64(hk)
        ov[pg.numpy(), :, (a % page).numpy()] = f64(hv)
    q, kn, vn = SI.gqa_prompt(sum(rows), seed=8)
    qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
    keep = [t.clone() for t in (qd, knd, vnd)]
    T, S = sum(rows), len(rows)
    max_ctx = max(p + r for p, r in zip(hist, rows))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    pl = torch.tensor(hist, dtype=torch.int32, device="cuda")
    ob, out = guarded((T, hq, d), torch.bfloat16)
    tb, td = guarded((3, max_blocks), torch.int32, table.cuda())
    ws = torch.zeros(cp.cp_workspace_size(desc, T, max_ctx, S), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_mixed_step(desc, qd, knd, vnd, kp, vp, td, cu, pl, S, T, max_ctx, out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bands_intact(ob) and bands_intact(kb) and bands_intact(vb) and bands_intact(tb)
    assert all(torch.equal(_bits(a), _bits(b)) for a, b in zip(keep, (qd, knd, vnd)))
    ref, ok, ov, newp = oracle.mixed_step(f64(q), f64(kn), f64(vn), ok, ov, table.numpy(), rows, hist)
    assert np.abs(f64(out) - ref).max() < BF16_TOL and pl.tolist() == newp
    mask = ~np.isnan(ok)
    got_k, got_v = f64(kp), f64(vp)
    assert np.array_equal(got_k[mask], ok[mask]) and np.isnan(got_k[~mask]).all()
    assert np.array_equal(got_v[mask], ov[mask]) and np.isnan(got_v[~mask]).all()


def test_varlen_call_stays_in_its_rows():
    """Ragged prompts in one call (one-row sequence on the split-KV path, the
    rest on the tensor-core kernel with its work list): bands intact."""
    hq, hkv, d, cap = 32, 8, 128, 1024
    pasts, rows = [0, 300, 511, 37], [200, 130, 1, 64]
    B = len(pasts)
    desc = cp.layer_desc(torch.bfloat16, B, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=cap)
    kb, kc = guarded((B, hkv, cap, d), torch.bfloat16, float("nan"))
    vb, vc = guarded((B, hkv, cap, d), torch.bfloat16, float("nan"))
    hist = []
    for s, p in enumerate(pasts):
        hk, hv = SI.normal((p, hkv, d), 40 + s).bfloat16(), SI.normal((p, hkv, d), 50 + s).bfloat16()
        kc[s, :, :p] = hk.permute(1, 0, 2).cuda()
        vc[s, :, :p] = hv.permute(1, 0, 2).cuda()
        hist.append((hk, hv))
    T = sum(rows)
    q, kn, vn = SI.gqa_prompt(T, seed=12)
    qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
    keep = [t.clone() for t in (qd, knd, vnd)]
    max_ctx = max(p + r for p, r in zip(pasts, rows))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    lens = torch.tensor(pasts, dtype=torch.int32, device="cuda")
    ob, out = guarded((T, hq, d), torch.bfloat16)
    wsz = cp.cp_workspace_size(desc, T, max_ctx, B)
    wb, ws16 = guarded(((wsz + 1) // 2,), torch.int16, 0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_prefill_varlen(desc, qd, knd, vnd, kc, vc, cu, lens, B, T, max_ctx, out, ws16.view(torch.uint8),
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and lens.tolist() == [p + r for p, r in zip(pasts, rows)]
    assert bands_intact(ob) and bands_intact(kb) and bands_intact(vb) and bands_intact(wb)
    assert all(torch.equal(_bits(a), _bits(b)) for a, b in zip(keep, (qd, knd, vnd)))
    o = f64(out)
    r0 = 0
    for s, (p, r) in enumerate(zip(pasts, rows)):
        keys = np.concatenate([f64(hist[s][0]), f64(kn[r0:r0 + r])])
        vals = np.concatenate([f64(hist[s][1]), f64(vn[r0:r0 + r])])
        ref = oracle.chunk_attention(f64(q[r0:r0 + r]), keys, vals, p)
        assert np.abs(o[r0:r0 + r] - ref).max() < BF16_TOL, s
        assert torch.isnan(kc[s, :, p + r:].float()).all()
        r0 += r


def test_pad_chunk_stays_in_its_rows():
    """The padding widening writes only rows [real, padded) of each sequence."""
    B, R, real, h, d = 3, 171, 100, 8, 128
    tensors = []
    for seed in range(3):
        x = SI.normal((B, R, h, d), 20 + seed).bfloat16().cuda()
        buf, view = guarded((B, R, h, d), torch.bfloat16, x)
        tensors.append((buf, view, x))
    desc = cp.layer_desc(torch.bfloat16, B, h, h, d, cp.CP_CACHE_CONTIG, capacity=256)
    cp.cp_pad_chunk(desc, tensors[0][1], tensors[1][1], tensors[2][1], real, R)
    torch.cuda.synchronize()
    for buf, view, x in tensors:
        assert bands_intact(buf)
        assert torch.equal(_bits(view[:, :real]), _bits(x[:, :real]))
        assert torch.equal(_bits(view[:, real:]), _bits(x[:, real - 1:real].expand(B, R - real, h, d)))
