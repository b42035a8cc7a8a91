"""GPU parity of cp_prefill_varlen: several sequences with ragged rows and
different cached lengths over one contiguous cache in a single call (the
glossary's step filled with chunks of several prompts), against the C++
oracle, with the cache checked byte for byte and each sequence's rows
bit-identical to the same sequence run alone."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import synth_inputs as SI
from gpu_util import BF16_TOL, f64
from oracle import cpp as oracle

pytestmark = pytest.mark.gpu

HQ, HKV, D, CAP = 32, 8, 128, 2048


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _setup(pasts, seed):
    """Cache [B, HKV, CAP, D] poisoned with NaN, positions [0, past) of each
    sequence filled with seeded history."""
    B = len(pasts)
    kc = torch.full((B, HKV, CAP, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    hist = []
    for s, p in enumerate(pasts):
        hk = SI.normal((p, HKV, D), seed + 2 * s)
        hv = SI.normal((p, HKV, D), seed + 2 * s + 1)
        kc[s, :, :p] = hk.permute(1, 0, 2).cuda()
        vc[s, :, :p] = hv.permute(1, 0, 2).cuda()
        hist.append((hk, hv))
    return kc, vc, hist


def _partials_bytes(B, max_ctx):
    """The split-KV partials a ragged call keeps at the start of its workspace."""
    return B * HQ * (-(-max_ctx // 512)) * (D + 2) * 4


def _call(kc, vc, pasts, rows, q, kn, vn, ws_bytes=None, keep_ws=False):
    B = len(pasts)
    desc = cp.layer_desc(torch.bfloat16, kc.shape[0], HQ, HKV, D, cp.CP_CACHE_CONTIG, capacity=CAP)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    lens = torch.tensor(pasts, dtype=torch.int32, device="cuda")
    T = int(sum(rows))
    max_ctx = max(p + r for p, r in zip(pasts, rows))
    out = torch.empty(T, HQ, D, dtype=torch.bfloat16, device="cuda")
    if ws_bytes is None:
        ws_bytes = cp.cp_workspace_size(desc, T, max_ctx, B)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_prefill_varlen(desc, q, kn, vn, kc, vc, cu, lens, B, T, max_ctx, out, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (out, lens, ws) if keep_ws else (out, lens)


@pytest.mark.parametrize("pasts,rows", [
    ([0, 37, 300, 1000, 128], [1, 5, 130, 257, 64]),
    ([1500, 0, 511], [300, 512, 2]),
])
def test_varlen_matches_oracle_and_runs_alone(pasts, rows):
    kc, vc, hist = _setup(pasts, seed=70)
    k0, v0 = kc.clone(), vc.clone()
    T = sum(rows)
    q, kn, vn = SI.gqa_prompt(T, seed=71)
    out, lens = _call(kc, vc, pasts, rows, q.cuda(), kn.cuda(), vn.cuda())
    assert lens.tolist() == [p + r for p, r in zip(pasts, rows)]
    o = f64(out)
    t = 0
    worst = 0.0
    for s, (p, r) in enumerate(zip(pasts, rows)):
        # the cache: history, then this call's rows, then the untouched poison
        got_k = kc[s].permute(1, 0, 2)
        assert torch.equal(got_k[:p].cpu(), hist[s][0]) and torch.equal(got_k[p:p + r].cpu(), kn[t:t + r])
        assert torch.equal(vc[s].permute(1, 0, 2)[p:p + r].cpu(), vn[t:t + r])
        assert torch.isnan(got_k[p + r:].float()).all()
        keys = np.concatenate([f64(hist[s][0]), f64(kn[t:t + r])])
        vals = np.concatenate([f64(hist[s][1]), f64(vn[t:t + r])])
        ref = oracle.chunk_attention(f64(q[t:t + r]), keys, vals, p)
        worst = max(worst, float(np.abs(o[t:t + r] - ref).max()))
        # the same sequence alone, from the same starting cache: bit-identical rows
        ks, vs = k0[s:s + 1].clone(), v0[s:s + 1].clone()
        alone, _ = _call(ks, vs, [p], [r], q[t:t + r].cuda(), kn[t:t + r].cuda(), vn[t:t + r].cuda())
        assert torch.equal(alone, out[t:t + r]), s
        t += r
    assert worst < BF16_TOL, worst


def test_work_list_is_heaviest_first_and_changes_no_bit():
    """The append kernel's work list for the tensor-core kernel holds every
    pair (64 tokens at G = 4) of every sequence with more than one row exactly
    once, ordered by the 128-key tiles its last token sees, most first, then
    empty entries.  A workspace with no room for the list (the split-KV
    partials only) takes the sequence-order scan instead, with bit-identical
    output: the list only changes which cluster computes which pair."""
    pasts, rows = [0, 1024, 1800, 512, 1900, 1, 100], [700, 300, 130, 257, 64, 1, 2]
    kc, vc, _ = _setup(pasts, seed=80)
    k0, v0 = kc.clone(), vc.clone()
    T, B = sum(rows), len(pasts)
    q, kn, vn = SI.gqa_prompt(T, seed=81)
    out, _, ws = _call(kc, vc, pasts, rows, q.cuda(), kn.cuda(), vn.cuda(), keep_ws=True)
    max_ctx = max(p + r for p, r in zip(pasts, rows))
    off = -(-_partials_bytes(B, max_ctx) // 16) * 16
    bound = -(-T // 64) + B
    lst = ws[off:off + 8 * bound].cpu().view(torch.int32).view(bound, 2).tolist()
    n_valid = sum(1 for s, _ in lst if s >= 0)
    assert all(s >= 0 for s, _ in lst[:n_valid]) and all(e == [-1, 0] for e in lst[n_valid:])
    want = sorted((s, k * 64) for s, r in enumerate(rows) if r > 1 for k in range(-(-r // 64)))
    got = [tuple(e) for e in lst[:n_valid]]
    assert sorted(got) == want

    def tiles(e):
        s, t0 = e
        return -(-(pasts[s] + min(t0 + 64, rows[s])) // 128)

    assert all(tiles(a) >= tiles(b) for a, b in zip(got, got[1:]))
    # no room for the list: the same rows, bit for bit
    kc.copy_(k0)
    vc.copy_(v0)
    plain, _ = _call(kc, vc, pasts, rows, q.cuda(), kn.cuda(), vn.cuda(), ws_bytes=_partials_bytes(B, max_ctx))
    assert torch.equal(plain, out)


def test_overlap_form_is_bit_identical_eager_and_captured():
    """cp_prefill_varlen_overlap (one-row sequences' split-KV kernels on a side
    stream beside the tensor-core kernel) gives cp_prefill_varlen's outputs,
    cache and lengths bit for bit, launched eagerly and replayed from a
    captured CUDA graph."""
    pasts, rows = [0, 37, 300, 1000, 128, 1500], [1, 5, 130, 257, 64, 1]
    T = sum(rows)
    q, kn, vn = (t.cuda() for t in SI.gqa_prompt(T, seed=81))
    desc = cp.layer_desc(torch.bfloat16, len(pasts), HQ, HKV, D, cp.CP_CACHE_CONTIG, capacity=CAP)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    max_ctx = max(p + r for p, r in zip(pasts, rows))
    base_k, base_v, _ = _setup(pasts, seed=80)

    def run(overlap, graph=False):
        kc, vc = base_k.clone(), base_v.clone()
        lens = torch.tensor(pasts, dtype=torch.int32, device="cuda")
        lens0 = lens.clone()
        out = torch.zeros(T, HQ, D, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(cp.cp_workspace_size(desc, T, max_ctx, len(pasts)), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        side, ev1, ev2 = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()

        def reset():
            kc.copy_(base_k)
            vc.copy_(base_v)
            lens.copy_(lens0)
            out.zero_()

        def call():
            if overlap:
                cp.cp_prefill_varlen_overlap(desc, q, kn, vn, kc, vc, cu, lens, len(pasts), T, max_ctx, out, ws,
                                             side, ev1, ev2, dev_status=status)
            else:
                cp.cp_prefill_varlen(desc, q, kn, vn, kc, vc, cu, lens, len(pasts), T, max_ctx, out, ws,
                                     dev_status=status)
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                call()  # warm-up outside the capture
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            reset()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            reset()
            g.replay()
        else:
            call()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return out, kc, vc, lens

    ref = run(False)
    for graph in (False, True):
        got = run(True, graph)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[3], ref[3]), graph
        assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(got[2].view(torch.int16), ref[2].view(torch.int16))
