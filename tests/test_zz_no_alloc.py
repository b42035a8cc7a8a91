"""cp_mixed_step_noalloc: the mixed step for callers that cannot allocate device
memory (engines whose memory is reserved up front, plugins handed only their
tensors, code running where cudaMalloc is not allowed).  It must give the same
results as cp_mixed_step with a caller workspace, on consecutive calls that
reuse its fixed scratch, and refuse steps that do not fit that scratch.

This file is collected last so a failure here cannot hide other failures."""
import ctypes

import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import synth_inputs as SI

HQ, HKV, D, PAGE = 32, 8, 128, 16


def test_oversized_step_is_refused_before_any_gpu_work():
    """A step whose split-KV scratch exceeds the fixed array returns
    CP_ERR_WORKSPACE before anything is enqueued (runs without a GPU)."""
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()
    desc = cp.layer_desc(torch.bfloat16, 0, HQ, HKV, D, cp.CP_CACHE_PAGED, page_size=PAGE,
                         num_pages=40000, max_blocks=600)
    need = cp.cp_workspace_size(desc, 64, 8192, 64)
    assert need > cp.cp_noalloc_scratch_bytes()
    fake = 1 << 20
    st = cp.lib().cp_mixed_step_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, fake, fake,
                                        64, 64, 8192, fake, None, None)
    assert st == cp.CP_ERR_WORKSPACE


def _pool_state(seed):
    ctx = [40, 300, 513, 800, 1000]
    prompt = 350
    lengths = ctx + [prompt]
    need = [-(-(n + 8) // PAGE) for n in lengths]
    max_blocks, num_pages = max(need), sum(need)
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))
    table = torch.full((len(need), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    desc = cp.layer_desc(torch.bfloat16, 0, HQ, HKV, D, cp.CP_CACHE_PAGED, page_size=PAGE,
                         num_pages=num_pages, max_blocks=max_blocks)
    kp = torch.zeros(num_pages, HKV, PAGE, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    for s, c in enumerate(ctx):  # history of each decode: positions [0, c-1)
        a = torch.arange(c - 1)
        pages = table[s, a // PAGE].long()
        kp[pages, :, a % PAGE] = SI.normal((c - 1, HKV, D), seed + 10 + s).to("cuda", torch.bfloat16)
        vp[pages, :, a % PAGE] = SI.normal((c - 1, HKV, D), seed + 20 + s).to("cuda", torch.bfloat16)
    past = [c - 1 for c in ctx] + [0]
    return desc, kp, vp, table.cuda(), past


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_on_consecutive_calls():
    """Two calls in a row through both entry points: the outputs, pools and
    past lengths are bit-identical (both run the same kernels on the same
    inputs, with a fixed merge order).  The second call lists fewer and shorter
    sequences than the first, so it uses fewer split-KV partials laid out
    differently in the shared scratch: leftovers of the first call must not
    reach its results."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()
    desc, kp, vp, table, past = _pool_state(31)
    kp_b, vp_b = kp.clone(), vp.clone()
    past_a = torch.tensor(past, dtype=torch.int32, device="cuda")
    past_b = past_a.clone()
    status_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    status_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    S = len(past)
    prompt_q, prompt_k, prompt_v = SI.gqa_prompt(350, seed=32)
    start = 0
    # call 1: the five decodes (contexts up to 1000: two 512-key splits) and 200 prompt rows;
    # call 2: decodes 0 and 1 only (contexts 41 and 301: one split) and the next 150 prompt rows
    for step, (seqs, chunk) in enumerate([(list(range(S)), 200), ([0, 1, S - 1], 150)]):
        nd = len(seqs) - 1
        dq, dk, dv = SI.gqa_prompt(nd, seed=40 + step)
        q = torch.cat([dq, prompt_q[start:start + chunk]]).cuda()
        kn = torch.cat([dk, prompt_k[start:start + chunk]]).cuda()
        vn = torch.cat([dv, prompt_v[start:start + chunk]]).cuda()
        rows = [1] * nd + [chunk]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
        T = int(sum(rows))
        idx = torch.tensor(seqs, device="cuda")
        pa, pb = past_a[idx].contiguous(), past_b[idx].contiguous()
        tb = table[idx].contiguous()
        max_ctx = int(max(p + r for p, r in zip(pa.tolist(), rows)))
        out_a = torch.empty(T, HQ, D, dtype=torch.bfloat16, device="cuda")
        out_b = torch.full_like(out_a, float("nan"))
        ws = torch.empty(cp.cp_workspace_size(desc, T, max_ctx, len(seqs)), dtype=torch.uint8, device="cuda")
        cp.cp_mixed_step(desc, q, kn, vn, kp, vp, tb, cu, pa, len(seqs), T, max_ctx, out_a, ws,
                         dev_status=status_a)
        cp.cp_mixed_step_noalloc(desc, q, kn, vn, kp_b, vp_b, tb, cu, pb, len(seqs), T, max_ctx, out_b,
                                 dev_status=status_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), step
        assert torch.equal(pa, pb)
        past_a[idx] = pa
        past_b[idx] = pb
        start += chunk
    assert torch.equal(kp, kp_b) and torch.equal(vp, vp_b)
    assert torch.equal(past_a, past_b)
    assert int(status_a.item()) == 0 and int(status_b.item()) == 0
