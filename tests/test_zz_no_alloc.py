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
TOL = 2e-2  # the max-abs bound the other bf16 parity tests use


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
    for step, chunk in enumerate([200, 150]):  # two calls in a row, reusing the scratch
        dq, dk, dv = SI.gqa_prompt(S - 1, seed=40 + step)
        q = torch.cat([dq, prompt_q[start:start + chunk]]).cuda()
        kn = torch.cat([dk, prompt_k[start:start + chunk]]).cuda()
        vn = torch.cat([dv, prompt_v[start:start + chunk]]).cuda()
        rows = [1] * (S - 1) + [chunk]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
        T = int(sum(rows))
        max_ctx = int(max(p + r for p, r in zip(past_a.tolist(), rows)))
        out_a = torch.empty(T, HQ, D, dtype=torch.bfloat16, device="cuda")
        out_b = torch.full_like(out_a, float("nan"))
        ws = torch.empty(cp.cp_workspace_size(desc, T, max_ctx, S), dtype=torch.uint8, device="cuda")
        cp.cp_mixed_step(desc, q, kn, vn, kp, vp, table, cu, past_a, S, T, max_ctx, out_a, ws,
                         dev_status=status_a)
        cp.cp_mixed_step_noalloc(desc, q, kn, vn, kp_b, vp_b, table, cu, past_b, S, T, max_ctx, out_b,
                                 dev_status=status_b)
        torch.cuda.synchronize()
        err = (out_a.float() - out_b.float()).abs().max().item()
        assert err <= TOL, (step, err)
        assert torch.isfinite(out_b.float()).all()
        assert torch.equal(past_a, past_b)
        start += chunk
    assert torch.equal(kp, kp_b) and torch.equal(vp, vp_b)
    assert int(status_a.item()) == 0 and int(status_b.item()) == 0
