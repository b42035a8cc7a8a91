"""GPU parity of the right-aligned rolling cache path (fp16, 16 heads x 128,
C = 1024, c = 256) against the oracle's literal cat/slice cache and additive
-32768 mask."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _run_rolling(n_real, c, C, H, d, dtype, seed, fused=False):
    L = cp.cp_aligned_length(n_real, c)
    lp = L - n_real
    q, k, v = SI.rolling_prompt(L, seed=seed, heads=H, dim=d, dtype=dtype)
    desc = cp.layer_desc(dtype, 1, H, H, d, cp.CP_CACHE_ROLLING, capacity=C)
    kc = torch.full((1, H, C, d), float("nan"), dtype=dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    left = torch.tensor([lp], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(L, H, d, dtype=dtype, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.zeros(cp.cp_workspace_size(desc, c, C, 1), dtype=torch.uint8, device="cuda")
    ref_out, snaps = oracle.rolling_prefill(f64(q), f64(k), f64(v), c, C, lp)
    for ci in range(L // c):
        sl = slice(ci * c, (ci + 1) * c)
        if fused:
            cp.cp_prefill_chunk(desc, qd[None, sl], kd[None, sl], vd[None, sl], kc, vc, lens, c, c, ci * c,
                                out[None, sl], ws, left_pad=left, dev_status=status)
        else:
            cp.cp_kv_append(desc, kd[None, sl], vd[None, sl], c, kc, vc, lens, ci * c, dev_status=status)
            cp.cp_prefill_chunk_attn(desc, qd[None, sl], kc, vc, lens, c, c, ci * c, out[None, sl], None,
                                     commit=True, left_pad=left, dev_status=status)
        torch.cuda.synchronize()
        # De-rotate: logical slot j holds position a = n - C + j, stored at a mod C.
        n = (ci + 1) * c
        ok_k, ok_v = snaps[ci]
        j = np.arange(C)
        a = n - C + j
        keep = a >= 0
        phys = torch.from_numpy(a[keep] % C)
        assert torch.equal(kc[0, :, phys].cpu().double(), torch.from_numpy(ok_k[:, keep])), ci
        assert torch.equal(vc[0, :, phys].cpu().double(), torch.from_numpy(ok_v[:, keep])), ci
    assert int(status.item()) == 0 and int(lens.item()) == L
    got = f64(out)
    err = np.abs(got[lp:] - ref_out[lp:]).max()
    assert err < BF16_TOL, err
    # Left-pad query rows see no key: their value is unpinned, only finite.
    assert np.isfinite(got).all()
    return got, ref_out, lp, q, k, v


def test_rolling_sliding_window_2048():
    """L = 2048 > C = 1024 (2000 real tokens, 48 left-pad): from chunk 4 on the
    oldest KV is forgotten (sliding-window regime)."""
    _run_rolling(2000, 256, 1024, 16, 128, torch.float16, seed=3)


def test_rolling_no_overflow_768_equals_plain_prefill():
    """L = 768 <= C (700 real tokens, 68 left-pad): the result equals ordinary
    causal prefill over the 700 real tokens."""
    got, _, lp, q, k, v = _run_rolling(700, 256, 1024, 16, 128, torch.float16, seed=3)
    plain = oracle.causal_attention(f64(q[lp:]), f64(k[lp:]), f64(v[lp:]))
    assert np.abs(got[lp:] - plain).max() < BF16_TOL


def test_rolling_sliding_window_fused_call():
    """The same window through the one-call chunk entry point: identical to
    the append + attention calls, bit for bit."""
    got, _, lp, _, _, _ = _run_rolling(2000, 256, 1024, 16, 128, torch.float16, seed=3, fused=True)
    ref, _, _, _, _, _ = _run_rolling(2000, 256, 1024, 16, 128, torch.float16, seed=3)
    assert np.array_equal(got, ref)


def test_rolling_small_ragged():
    """A cache that is not a multiple of the 128-key tile, bf16, head_dim 64."""
    _run_rolling(300, 48, 176, 4, 64, torch.bfloat16, seed=11)


@pytest.mark.parametrize("n_real,c,C,H,d,dtype,seed", [
    (300, 48, 176, 4, 64, torch.bfloat16, 11),    # ring not a multiple of the tile, chunks of 48
    (700, 96, 384, 8, 128, torch.float16, 12),    # chunks of 96: the new slots straddle 128-slot tiles
    (1100, 256, 384, 4, 128, torch.bfloat16, 13), # chunks of 256 = capacity - 128: the widest split
])
def test_rolling_fused_equals_separate_at_straddling_chunks(n_real, c, C, H, d, dtype, seed):
    """One-call chunks on a ring (the kernel reads the chunk's slots from k_new,
    walks a tile that holds cached and new slots twice, and copies the rows
    into the ring): the oracle's outputs and ring contents, and the separate
    append + attention calls bit for bit."""
    got, _, lp, _, _, _ = _run_rolling(n_real, c, C, H, d, dtype, seed=seed, fused=True)
    ref, _, _, _, _, _ = _run_rolling(n_real, c, C, H, d, dtype, seed=seed)
    assert np.array_equal(got, ref)


def _run_gqa(c, fused):
    n_real, C, hq, hkv, d = 500, 384, 8, 2, 128
    G = hq // hkv
    L = cp.cp_aligned_length(n_real, c)
    lp = L - n_real
    q, _, _ = SI.rolling_prompt(L, seed=21, heads=hq, dim=d, dtype=torch.bfloat16)
    _, k, v = SI.rolling_prompt(L, seed=22, heads=hkv, dim=d, dtype=torch.bfloat16)
    desc = cp.layer_desc(torch.bfloat16, 1, hq, hkv, d, cp.CP_CACHE_ROLLING, capacity=C)
    kc = torch.full((1, hkv, C, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    left = torch.tensor([lp], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(L, hq, d, dtype=torch.bfloat16, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.zeros(cp.cp_workspace_size(desc, c, C, 1), dtype=torch.uint8, device="cuda")
    for ci in range(L // c):
        sl = slice(ci * c, (ci + 1) * c)
        if fused:
            cp.cp_prefill_chunk(desc, qd[None, sl], kd[None, sl], vd[None, sl], kc, vc, lens, c, c, ci * c,
                                out[None, sl], ws, left_pad=left, dev_status=status)
        else:
            cp.cp_kv_append(desc, kd[None, sl], vd[None, sl], c, kc, vc, lens, ci * c, dev_status=status)
            cp.cp_prefill_chunk_attn(desc, qd[None, sl], kc, vc, lens, c, c, ci * c, out[None, sl], None,
                                     commit=True, left_pad=left, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(lens.item()) == L
    k_rep = np.repeat(f64(k), G, axis=1)
    v_rep = np.repeat(f64(v), G, axis=1)
    ref, snaps = oracle.rolling_prefill(f64(q), k_rep, v_rep, c, C, lp)
    got = f64(out)
    assert np.abs(got[lp:] - ref[lp:]).max() < BF16_TOL
    assert np.isfinite(got).all()
    # final window: logical slot j holds position a = L - C + j, stored at a mod C
    ok_k, ok_v = snaps[-1]
    j = np.arange(C)
    a = L - C + j
    keep = a >= 0
    phys = torch.from_numpy(a[keep] % C)
    assert torch.equal(kc[0, :, phys].cpu().double(), torch.from_numpy(ok_k[::G][:, keep]))
    assert torch.equal(vc[0, :, phys].cpu().double(), torch.from_numpy(ok_v[::G][:, keep]))
    return got


def test_rolling_gqa():
    """Rolling window with grouped-query heads (8 query / 2 KV heads, bf16):
    compared with the oracle's rolling prefill on the K/V heads repeated per
    query head (grouped-query attention equals that multi-head attention)."""
    _run_gqa(128, fused=False)


@pytest.mark.parametrize("c", [128, 96])
def test_rolling_gqa_fused_call(c):
    """The same grouped-query window through the one-call chunk entry point
    (chunks of 96 put the new slots across 128-slot tiles): the oracle, and
    the separate append + attention calls bit for bit."""
    assert np.array_equal(_run_gqa(c, fused=True), _run_gqa(c, fused=False))


def _run_ring_batch(n_reals, c, C, hq, hkv, d, dtype, seed, fused):
    """A batch of left-padded sequences of one aligned length on a ring cache,
    chunk by chunk; returns (out [B, L, hq, d] float64, k ring, v ring, L)."""
    L = max(cp.cp_aligned_length(n, c) for n in n_reals)
    B = len(n_reals)
    G = hq // hkv
    qs, ks, vs = [], [], []
    for b in range(B):
        q, _, _ = SI.rolling_prompt(L, seed=seed + 2 * b, heads=hq, dim=d, dtype=dtype)
        _, k, v = SI.rolling_prompt(L, seed=seed + 2 * b + 1, heads=hkv, dim=d, dtype=dtype)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    qd, kd, vd = (torch.stack(t).cuda() for t in (qs, ks, vs))
    desc = cp.layer_desc(dtype, B, hq, hkv, d, cp.CP_CACHE_ROLLING, capacity=C)
    kc = torch.full((B, hkv, C, d), float("nan"), dtype=dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    left = torch.tensor([L - n for n in n_reals], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(B, L, hq, d, dtype=dtype, device="cuda")
    ws = torch.zeros(cp.cp_workspace_size(desc, B * c, C, B), dtype=torch.uint8, device="cuda")
    for ci in range(L // c):
        sl = slice(ci * c, (ci + 1) * c)
        q_, k_, v_ = qd[:, sl].contiguous(), kd[:, sl].contiguous(), vd[:, sl].contiguous()
        o_ = torch.empty_like(q_)
        if fused:
            cp.cp_prefill_chunk(desc, q_, k_, v_, kc, vc, lens, c, c, ci * c, o_, ws, left_pad=left,
                                dev_status=status)
        else:
            cp.cp_kv_append(desc, k_, v_, c, kc, vc, lens, ci * c, dev_status=status)
            cp.cp_prefill_chunk_attn(desc, q_, kc, vc, lens, c, c, ci * c, o_, None, commit=True,
                                     left_pad=left, dev_status=status)
        out[:, sl] = o_
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(lens.cpu(), torch.full((B,), L, dtype=torch.int32))
    got = f64(out)
    assert np.isfinite(got).all()
    j = np.arange(C)
    a = L - C + j
    keep = a >= 0
    phys = torch.from_numpy(a[keep] % C)
    for b, n in enumerate(n_reals):
        lp = L - n
        k_rep = np.repeat(f64(ks[b]), G, axis=1)
        v_rep = np.repeat(f64(vs[b]), G, axis=1)
        ref, snaps = oracle.rolling_prefill(f64(qs[b]), k_rep, v_rep, c, C, lp)
        err = np.abs(got[b, lp:] - ref[lp:]).max()
        assert err < BF16_TOL, (b, err)
        ok_k, ok_v = snaps[-1]
        assert torch.equal(kc[b, :, phys].cpu().double(), torch.from_numpy(ok_k[::G][:, keep])), b
        assert torch.equal(vc[b, :, phys].cpu().double(), torch.from_numpy(ok_v[::G][:, keep])), b
    return got


@pytest.mark.parametrize("n_reals,c,C,hq,hkv,d,dtype", [
    ((700, 650), 128, 384, 8, 2, 128, torch.bfloat16),   # two sequences, left pads 68 and 118
    ((500, 333, 480), 96, 352, 4, 4, 64, torch.float16),  # three sequences, MHA, head_dim 64
    ((450,), 64, 256, 16, 2, 64, torch.bfloat16),        # GQA 8, head_dim 64
    ((300,), 64, 320, 16, 1, 128, torch.float16),        # GQA 16 (one KV head)
])
def test_rolling_batches_and_groups(n_reals, c, C, hq, hkv, d, dtype):
    """Ring caches for a batch of left-padded sequences and for large query
    groups: each sequence against the oracle's rolling prefill (K/V heads
    repeated per query head) with its ring de-rotated byte for byte, through
    the one-call entry point and the separate calls, bit for bit."""
    fused = _run_ring_batch(n_reals, c, C, hq, hkv, d, dtype, seed=40, fused=True)
    split = _run_ring_batch(n_reals, c, C, hq, hkv, d, dtype, seed=40, fused=False)
    assert np.array_equal(fused, split)
