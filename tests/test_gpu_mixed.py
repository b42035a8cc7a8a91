"""GPU parity of the token-budget mixed step over a paged cache (decode rows
on the split-KV path, prompt chunks on the tensor-core path) against the
oracle, plus batch invariance."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI
from gpu_util import BF16_TOL, f64

pytestmark = pytest.mark.gpu

HQ, HKV, D, PAGE = 32, 8, 128, 16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


class Paged:
    """GPU pools + an oracle copy of the same pools."""

    def __init__(self, mb: SI.MixedBatch, with_oracle=True, dtype=torch.bfloat16):
        self.mb = mb
        self.dtype = dtype
        self.desc = cp.layer_desc(dtype, 0, HQ, HKV, D, cp.CP_CACHE_PAGED, page_size=mb.page_size,
                                  num_pages=mb.num_pages, max_blocks=mb.max_blocks)
        self.k = torch.full((mb.num_pages, HKV, mb.page_size, D), float("nan"), dtype=dtype, device="cuda")
        self.v = torch.full_like(self.k, float("nan"))
        self.table = mb.block_table.cuda()
        self.ok = np.full(tuple(self.k.shape), np.nan) if with_oracle else None
        self.ov = np.full(tuple(self.k.shape), np.nan) if with_oracle else None
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def prefill_history(self, s, kv_k, kv_v):
        """Write positions [0, n) of sequence s directly (test set-up)."""
        n = kv_k.shape[0]
        a = torch.arange(n)
        pages = self.mb.block_table[s, a // PAGE].long()
        self.k[pages, :, a % PAGE] = kv_k.to("cuda", self.dtype)
        self.v[pages, :, a % PAGE] = kv_v.to("cuda", self.dtype)
        if self.ok is not None:
            self.ok[pages.numpy(), :, (a % PAGE).numpy()] = f64(kv_k.to(self.dtype))
            self.ov[pages.numpy(), :, (a % PAGE).numpy()] = f64(kv_v.to(self.dtype))

    def args(self, seqs, rows, past, max_ctx):
        """Device buffers of one step: cu_rows, past lengths, block table, output, workspace."""
        S = len(seqs)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
        pl = torch.tensor(past, dtype=torch.int32, device="cuda")
        bt = self.table[torch.tensor(seqs, device="cuda")].contiguous()
        T = int(sum(rows))
        out = torch.empty(T, HQ, D, dtype=self.dtype, device="cuda")
        ws = torch.zeros(cp.cp_workspace_size(self.desc, T, max_ctx, S), dtype=torch.uint8, device="cuda")
        return cu, pl, bt, out, ws

    def launch(self, q, kn, vn, cu, pl, bt, out, ws, max_ctx, overlap=None):
        """One step on the current stream; `overlap` = (side stream, fork event, join event)."""
        S, T = pl.numel(), q.shape[0]
        if overlap is None:
            cp.cp_mixed_step(self.desc, q, kn, vn, self.k, self.v, bt, cu, pl, S, T, max_ctx, out, ws,
                             dev_status=self.status)
        else:
            cp.cp_mixed_step_overlap(self.desc, q, kn, vn, self.k, self.v, bt, cu, pl, S, T, max_ctx, out, ws,
                                     *overlap, dev_status=self.status)

    def step(self, seqs, rows, past, q, kn, vn, max_ctx, overlap=None):
        cu, pl, bt, out, ws = self.args(seqs, rows, past, max_ctx)
        self.launch(q, kn, vn, cu, pl, bt, out, ws, max_ctx, overlap)
        return out, pl


def _schedule_steps(budget, n_dec, prompts):
    steps = {}
    for st, seq, start, r in cp.cp_schedule(budget, n_dec, prompts):
        steps.setdefault(st, []).append((seq, start, r))
    return [steps[i] for i in sorted(steps)]


def _layout(ctx, prompts, seed):
    """A MixedBatch for the given decode contexts and prompt lengths, pages from a seeded permutation."""
    mb = SI.mixed_batch(n_decode=len(ctx), ctx_lo=1, ctx_hi=2, n_prompt=len(prompts), prompt_len=prompts[0],
                        decode_tail=64, seed=seed)
    mb.decode_ctx = list(ctx)
    mb.prompt_lens = list(prompts)
    need = [-(-(n + 64) // PAGE) for n in list(ctx) + list(prompts)]
    mb.max_blocks = max(need)
    mb.num_pages = sum(need)
    perm = torch.randperm(mb.num_pages, generator=torch.Generator().manual_seed(seed))
    mb.block_table = torch.full((len(need), mb.max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        mb.block_table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    return mb


def _same_bits(a, b):
    """Equal bit patterns (pool slots never written hold NaN)."""
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _overlap_handles():
    return torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()


def _run_schedule(budget, ctx, prompts, seed, overlap=False):
    """Every step cp_schedule gives for `budget`, on the GPU and in the oracle:
    each step's every row within tolerance, past lengths advanced by the rows,
    and at the end the pools equal the oracle's bit for bit (slots never
    written stay NaN).  Returns the number of steps."""
    mb = _layout(ctx, prompts, seed)
    P = Paged(mb)
    pos = [c - 1 for c in ctx] + [0] * len(prompts)
    for s, c in enumerate(ctx):
        if c > 1:
            P.prefill_history(s, SI.normal((c - 1, HKV, D), 100 + s), SI.normal((c - 1, HKV, D), 200 + s))
    pq = [SI.gqa_prompt(n, seed=30 + i) for i, n in enumerate(prompts)]
    nd = len(ctx)
    plan = _schedule_steps(budget, nd, prompts)
    handles = _overlap_handles() if overlap else None
    for si, entries in enumerate(plan):
        assert sum(r for _, _, r in entries) <= budget
        seqs, rows, qs, ks, vs = [], [], [], [], []
        for seq, start, r in entries:
            seqs.append(seq)
            rows.append(r)
            if start < 0:  # a decode row: fresh token
                t = SI.gqa_prompt(1, seed=1000 * si + seq)
                qs.append(t[0]); ks.append(t[1]); vs.append(t[2])
            else:
                q_, k_, v_ = pq[seq - nd]
                qs.append(q_[start:start + r]); ks.append(k_[start:start + r]); vs.append(v_[start:start + r])
        q = torch.cat(qs); kn = torch.cat(ks); vn = torch.cat(vs)
        past = [pos[s] for s in seqs]
        max_ctx = max(p + r for p, r in zip(past, rows))
        out, pl = P.step(seqs, rows, past, q.cuda(), kn.cuda(), vn.cuda(), max_ctx, handles)
        torch.cuda.synchronize()
        ref, P.ok, P.ov, newp = oracle.mixed_step(f64(q), f64(kn), f64(vn), P.ok, P.ov,
                                                  mb.block_table[seqs].numpy(), rows, past)
        err = np.abs(f64(out) - ref).max()
        assert err < BF16_TOL, (si, err)
        assert pl.tolist() == newp
        for s, p in zip(seqs, newp):
            pos[s] = p
    assert int(P.status.item()) == 0
    for got, want in ((f64(P.k), P.ok), (f64(P.v), P.ov)):
        mask = ~np.isnan(want)
        assert np.array_equal(got[mask], want[mask])
        assert np.isnan(got[~mask]).all()
    assert all(pos[nd + i] >= n for i, n in enumerate(prompts))  # every prompt was scheduled in full
    return len(plan)


def test_mixed_steps_reduced_full_check():
    """8 decodes with contexts at page and split edges plus 2 prompts, budget 256."""
    n = _run_schedule(256, [1, 2, 16, 17, 511, 512, 513, 700], [600, 450], seed=21)
    assert n >= 5


def test_overlap_schedule_reduced_full_check():
    """The same schedule through cp_mixed_step_overlap (split-KV kernels on a
    side stream): every row against the oracle, then the pools."""
    n = _run_schedule(256, [1, 2, 16, 17, 511, 512, 513, 700], [600, 450], seed=21, overlap=True)
    assert n >= 5


def test_overlap_is_bit_identical_to_mixed_step():
    """64 decodes (contexts U{1..3000}) beside a 1500-row prompt chunk:
    cp_mixed_step_overlap gives cp_mixed_step's output, pools and lengths bit
    for bit, launched eagerly and replayed from a captured CUDA graph."""
    ctx = torch.randint(1, 3001, (64,), generator=torch.Generator().manual_seed(31)).tolist()
    mb = _layout(ctx, [1500], seed=31)
    P = Paged(mb, with_oracle=False)
    for s, c in enumerate(ctx):
        if c > 1:
            P.prefill_history(s, SI.normal((c - 1, HKV, D), 700 + s), SI.normal((c - 1, HKV, D), 800 + s))
    dq, dk, dv = SI.gqa_prompt(64, seed=52)
    qp, kp, vp = SI.gqa_prompt(1500, seed=53)
    q = torch.cat([dq, qp]).cuda(); kn = torch.cat([dk, kp]).cuda(); vn = torch.cat([dv, vp]).cuda()
    seqs, rows, past = list(range(65)), [1] * 64 + [1500], [c - 1 for c in ctx] + [0]
    max_ctx = max(p + r for p, r in zip(past, rows))
    k0, v0 = P.k.clone(), P.v.clone()
    want, pl_want = P.step(seqs, rows, past, q, kn, vn, max_ctx)
    torch.cuda.synchronize()
    kw, vw = P.k.clone(), P.v.clone()
    handles = _overlap_handles()
    P.k.copy_(k0); P.v.copy_(v0)
    got, pl_got = P.step(seqs, rows, past, q, kn, vn, max_ctx, handles)
    torch.cuda.synchronize()
    assert torch.equal(got, want) and torch.equal(pl_got, pl_want)
    assert _same_bits(P.k, kw) and _same_bits(P.v, vw)
    # Captured: both streams join back into the capture stream.
    cu, pl, bt, out, ws = P.args(seqs, rows, past, max_ctx)
    past_dev = pl.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        P.launch(q, kn, vn, cu, pl, bt, out, ws, max_ctx, handles)
    for _ in range(2):
        P.k.copy_(k0); P.v.copy_(v0); pl.copy_(past_dev); out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want) and torch.equal(pl, pl_want)
        assert _same_bits(P.k, kw) and _same_bits(P.v, vw)
    assert int(P.status.item()) == 0


def test_mixed_schedule_budget_2048():
    """The budget-2048 schedule of the mixed workload at reduced sizes: 64
    running decodes (contexts U{1..600}) and 4 prompts of 1500 tokens; every
    step of the whole schedule is checked row by row, then the pools."""
    ctx = torch.randint(1, 601, (64,), generator=torch.Generator().manual_seed(23)).tolist()
    n = _run_schedule(2048, ctx, [1500] * 4, seed=23)
    assert n == 4  # 6000 prompt tokens at 2048 - 64 per step


def test_mixed_step_batch_invariance():
    """A request's rows are bit-identical whether it runs in a full mixed step
    or alone (fixed split length, tiles aligned to each sequence's start)."""
    ctx = [900, 37, 2000]
    mb = SI.mixed_batch(n_decode=3, ctx_lo=1, ctx_hi=2, n_prompt=1, prompt_len=700, seed=22)
    need = [-(-(n + 64) // PAGE) for n in ctx + [700]]
    mb.max_blocks, mb.num_pages = max(need), sum(need)
    mb.block_table = torch.full((4, mb.max_blocks), -1, dtype=torch.int32)
    perm = torch.randperm(mb.num_pages, generator=torch.Generator().manual_seed(5))
    off = 0
    for s, nb in enumerate(need):
        mb.block_table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    P = Paged(mb, with_oracle=False)
    for s, c in enumerate(ctx):
        P.prefill_history(s, SI.normal((c - 1, HKV, D), 300 + s), SI.normal((c - 1, HKV, D), 400 + s))
    qp, kp, vp = SI.gqa_prompt(700, seed=44)
    dq, dk, dv = SI.gqa_prompt(3, seed=45)
    q = torch.cat([dq, qp[:300]]).cuda()
    kn = torch.cat([dk, kp[:300]]).cuda()
    vn = torch.cat([dv, vp[:300]]).cuda()
    k0, v0 = P.k.clone(), P.v.clone()
    full, _ = P.step([0, 1, 2, 3], [1, 1, 1, 300], [c - 1 for c in ctx] + [0], q, kn, vn, 2000)
    torch.cuda.synchronize()
    for sel, rows_sel in [([1], slice(1, 2)), ([3], slice(3, 303)), ([2, 3], slice(2, 303))]:
        P.k.copy_(k0); P.v.copy_(v0)
        rows = [1 if s < 3 else 300 for s in sel]
        past = [(ctx[s] - 1) if s < 3 else 0 for s in sel]
        alone, _ = P.step(sel, rows, past, q[rows_sel].contiguous(), kn[rows_sel].contiguous(),
                          vn[rows_sel].contiguous(), 2000)
        torch.cuda.synchronize()
        assert torch.equal(alone, full[rows_sel]), sel
    assert int(P.status.item()) == 0


def test_mixed_step_full_size_first_step():
    """The mixed-step workload at full size: 64 decodes with contexts
    U{512..8192} in 16-token pages plus the first 8128-row chunk of a
    20000-token prompt (budget 8192).  All 64 decode rows and 64 sampled
    prompt rows match the oracle one by one."""
    mb = SI.mixed_batch()
    P = Paged(mb, with_oracle=False)
    hist = []
    for s, c in enumerate(mb.decode_ctx):
        hk, hv = SI.normal((c - 1, HKV, D), 500 + s), SI.normal((c - 1, HKV, D), 600 + s)
        P.prefill_history(s, hk, hv)
        hist.append((hk, hv))
    entries = _schedule_steps(8192, 64, mb.prompt_lens)[0]
    assert entries[-1] == (64, 0, 8128)
    qp, kp, vp = SI.gqa_prompt(8128, seed=50)
    dq, dk, dv = SI.gqa_prompt(64, seed=51)
    seqs = list(range(65))
    rows = [1] * 64 + [8128]
    past = [c - 1 for c in mb.decode_ctx] + [0]
    q = torch.cat([dq, qp]).cuda(); kn = torch.cat([dk, kp]).cuda(); vn = torch.cat([dv, vp]).cuda()
    out, pl = P.step(seqs, rows, past, q, kn, vn, max(8192, 8128))
    torch.cuda.synchronize()
    assert int(P.status.item()) == 0
    assert pl.tolist() == [p + r for p, r in zip(past, rows)]
    o = f64(out)
    worst = 0.0
    for s in range(64):
        ks = np.concatenate([f64(hist[s][0].to(torch.bfloat16)), f64(dk[s:s + 1])])
        vs = np.concatenate([f64(hist[s][1].to(torch.bfloat16)), f64(dv[s:s + 1])])
        ref = oracle.attention_row(f64(dq[s]), ks, vs, past[s])
        worst = max(worst, np.abs(o[s] - ref).max())
    rng = np.random.default_rng(1)
    kk, vv, qq = f64(kp), f64(vp), f64(qp)
    for p in [0, 1, 127, 128, 8127] + list(rng.integers(0, 8128, 59)):
        ref = oracle.attention_row(qq[p], kk, vv, int(p))
        worst = max(worst, np.abs(o[64 + p] - ref).max())
    assert worst < BF16_TOL, worst


def test_bad_page_id_is_reported_not_read():
    """A block-table entry outside the pool is never dereferenced; the step
    flags CP_DEV_BOUNDS in the device status word."""
    mb = SI.mixed_batch(n_decode=2, ctx_lo=40, ctx_hi=40, n_prompt=1, prompt_len=64, seed=23)
    P = Paged(mb, with_oracle=False)
    P.table[0, 1] = mb.num_pages + 5  # page of positions 16..31 of sequence 0
    q, kn, vn = SI.gqa_prompt(2 + 64, seed=46)
    out, _ = P.step([0, 1, 2], [1, 1, 64], [39, 39, 0], q.cuda(), kn.cuda(), vn.cuda(), 64)
    torch.cuda.synchronize()
    assert int(P.status.item()) & cp.CP_DEV_BOUNDS


def _decode_only_batch(ctx, seed):
    mb = SI.mixed_batch(n_decode=len(ctx), ctx_lo=1, ctx_hi=2, n_prompt=1, prompt_len=64, decode_tail=64,
                        seed=seed)
    mb.decode_ctx = list(ctx)
    need = [-(-(n + 64) // PAGE) for n in ctx]
    mb.max_blocks, mb.num_pages = max(need), sum(need)
    perm = torch.randperm(mb.num_pages, generator=torch.Generator().manual_seed(seed))
    mb.block_table = torch.full((len(need), mb.max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        mb.block_table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    return mb


def test_all_decode_steps_match_oracle():
    """Steps made only of decode rows (one row per sequence: the tensor-core
    path is not launched) at contexts on page and 512-key split edges, two
    steps in a row: every row matches the oracle's mixed step and the pools
    match it bit for bit."""
    ctx = [1, 2, 16, 511, 512, 513, 1024, 1025, 3000, 77]
    mb = _decode_only_batch(ctx, seed=24)
    P = Paged(mb)
    for s, c in enumerate(ctx):
        P.prefill_history(s, SI.normal((c - 1, HKV, D), 700 + s), SI.normal((c - 1, HKV, D), 800 + s))
    seqs = list(range(len(ctx)))
    rows = [1] * len(ctx)
    past = [c - 1 for c in ctx]
    for step in range(2):
        q, kn, vn = SI.gqa_prompt(len(ctx), seed=60 + step)
        out, pl = P.step(seqs, rows, past, q.cuda(), kn.cuda(), vn.cuda(), max(past) + 1)
        torch.cuda.synchronize()
        ref, P.ok, P.ov, newp = oracle.mixed_step(f64(q), f64(kn), f64(vn), P.ok, P.ov,
                                                  mb.block_table[seqs].numpy(), rows, past)
        err = np.abs(f64(out) - ref).max()
        assert err < BF16_TOL, (step, err)
        assert pl.tolist() == newp
        past = newp
    assert int(P.status.item()) == 0
    got_k = f64(P.k)
    mask = ~np.isnan(P.ok)
    assert np.array_equal(got_k[mask], P.ok[mask])


def test_sequence_without_rows_is_reported():
    """A mixed step lists only sequences with rows; a listed sequence with no
    rows is reported in the device status word."""
    ctx = [40, 300, 90]
    mb = _decode_only_batch(ctx, seed=25)
    P = Paged(mb, with_oracle=False)
    for s, c in enumerate(ctx):
        P.prefill_history(s, SI.normal((c - 1, HKV, D), 900 + s), SI.normal((c - 1, HKV, D), 950 + s))
    q, kn, vn = SI.gqa_prompt(3, seed=62)
    P.step([0, 1, 2], [0, 2, 1], [39, 299, 89], q.cuda(), kn.cuda(), vn.cuda(), 301)
    torch.cuda.synchronize()
    assert int(P.status.item()) & cp.CP_DEV_BOUNDS


@pytest.mark.parametrize("page", [32, 64, 128])
def test_mixed_step_page_sizes(page):
    """One mixed step (decode rows at page and split edges plus a prompt
    chunk) with 32-, 64- and 128-token pages: every row matches the oracle and
    the pools match it bit for bit."""
    ctx = [page, page + 1, 513, 1100]
    prompt = 300
    n_dec = len(ctx)
    need = [-(-(n + 64) // page) for n in ctx + [prompt]]
    max_blocks, num_pages = max(need), sum(need)
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(page))
    table = torch.full((len(need), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    desc = cp.layer_desc(torch.bfloat16, 0, HQ, HKV, D, cp.CP_CACHE_PAGED, page_size=page,
                         num_pages=num_pages, max_blocks=max_blocks)
    kp = torch.full((num_pages, HKV, page, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    ok = np.full(tuple(kp.shape), np.nan)
    ov = np.full(tuple(kp.shape), np.nan)
    for s, c in enumerate(ctx):  # history: positions [0, c - 1)
        hk, hv = SI.normal((c - 1, HKV, D), 1200 + s), SI.normal((c - 1, HKV, D), 1300 + s)
        a = torch.arange(c - 1)
        pg = table[s, a // page].long()
        kp[pg, :, a % page] = hk.to("cuda", torch.bfloat16)
        vp[pg, :, a % page] = hv.to("cuda", torch.bfloat16)
        ok[pg.numpy(), :, (a % page).numpy()] = f64(hk.to(torch.bfloat16))
        ov[pg.numpy(), :, (a % page).numpy()] = f64(hv.to(torch.bfloat16))
    dq, dk, dv = SI.gqa_prompt(n_dec, seed=70 + page)
    pq, pk, pv = SI.gqa_prompt(prompt, seed=71 + page)
    q = torch.cat([dq, pq]); kn = torch.cat([dk, pk]); vn = torch.cat([dv, pv])
    rows = [1] * n_dec + [prompt]
    past = [c - 1 for c in ctx] + [0]
    S, T = len(rows), sum(rows)
    max_ctx = max(p + r for p, r in zip(past, rows))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    pl = torch.tensor(past, dtype=torch.int32, device="cuda")
    out = torch.empty(T, HQ, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(cp.cp_workspace_size(desc, T, max_ctx, S), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_mixed_step(desc, q.cuda(), kn.cuda(), vn.cuda(), kp, vp, table.cuda(), cu, pl, S, T, max_ctx, out, ws,
                     dev_status=status)
    torch.cuda.synchronize()
    ref, ok, ov, newp = oracle.mixed_step(f64(q), f64(kn), f64(vn), ok, ov, table.numpy(), rows, past)
    assert int(status.item()) == 0
    assert np.abs(f64(out) - ref).max() < BF16_TOL
    assert pl.tolist() == newp
    got_k, got_v = f64(kp), f64(vp)
    mask = ~np.isnan(ok)
    assert np.array_equal(got_k[mask], ok[mask]) and np.array_equal(got_v[mask], ov[mask])


@pytest.mark.parametrize("page,dtype,hq,hkv,d", [
    (16, torch.bfloat16, 32, 8, 128),
    (32, torch.float16, 32, 8, 128),
    (64, torch.bfloat16, 16, 2, 128),
    (128, torch.float16, 8, 8, 128),
    (16, torch.float16, 16, 16, 128),
    (16, torch.bfloat16, 32, 8, 64),
])
def test_prompt_chunk_over_cached_pages(page, dtype, hq, hkv, d):
    """A prompt chunk whose keys are mostly cached pages (the tensor-core path
    reads them page by page; at head_dim 128 one box per page in the page
    layout), beside two decode rows: a first prompt of 700 tokens is already in
    the pool, the step brings its next 200 rows.  Every row against the oracle,
    the pools bit for bit."""
    ctx = [301, 1030]
    past_p, R = 700, 200
    lens = ctx + [past_p + R]
    need = [-(-(n + 64) // page) for n in lens]
    max_blocks, num_pages = max(need), sum(need)
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(page + hq))
    table = torch.full((len(need), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[off:off + nb].to(torch.int32)
        off += nb
    desc = cp.layer_desc(dtype, 0, hq, hkv, d, cp.CP_CACHE_PAGED, page_size=page, num_pages=num_pages,
                         max_blocks=max_blocks)
    kp = torch.full((num_pages, hkv, page, d), float("nan"), dtype=dtype, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    ok = np.full(tuple(kp.shape), np.nan)
    ov = np.full(tuple(kp.shape), np.nan)
    hist = [c - 1 for c in ctx] + [past_p]
    for s, n in enumerate(hist):  # positions [0, n) already in the pool
        hk, hv = SI.normal((n, hkv, d), 1400 + s).to(dtype), SI.normal((n, hkv, d), 1500 + s).to(dtype)
        a = torch.arange(n)
        pg = table[s, a // page].long()
        kp[pg, :, a % page] = hk.cuda()
        vp[pg, :, a % page] = hv.cuda()
        ok[pg.numpy(), :, (a % page).numpy()] = f64(hk)
        ov[pg.numpy(), :, (a % page).numpy()] = f64(hv)
    dq, dk, dv = SI.gqa_prompt(2, seed=80 + page, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    pq, pk, pv = SI.gqa_prompt(R, seed=81 + page, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    q = torch.cat([dq, pq]); kn = torch.cat([dk, pk]); vn = torch.cat([dv, pv])
    rows = [1, 1, R]
    S, T = len(rows), sum(rows)
    max_ctx = max(p + r for p, r in zip(hist, rows))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(rows)]), dtype=torch.int32, device="cuda")
    pl = torch.tensor(hist, dtype=torch.int32, device="cuda")
    out = torch.empty(T, hq, d, dtype=dtype, device="cuda")
    ws = torch.zeros(cp.cp_workspace_size(desc, T, max_ctx, S), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cp.cp_mixed_step(desc, q.cuda(), kn.cuda(), vn.cuda(), kp, vp, table.cuda(), cu, pl, S, T, max_ctx, out, ws,
                     dev_status=status)
    torch.cuda.synchronize()
    ref, ok, ov, newp = oracle.mixed_step(f64(q), f64(kn), f64(vn), ok, ov, table.numpy(), rows, hist)
    assert int(status.item()) == 0
    err = np.abs(f64(out) - ref).max()
    assert err < BF16_TOL, err
    assert pl.tolist() == newp
    got_k, got_v = f64(kp), f64(vp)
    mask = ~np.isnan(ok)
    assert np.array_equal(got_k[mask], ok[mask]) and np.array_equal(got_v[mask], ov[mask])
    assert np.isnan(got_k[~mask]).all() and np.isnan(got_v[~mask]).all()
