"""The C-ABI library on the CPU: it loads, exports every function that
include/cp_api.h declares, its integer helpers equal the oracle's, and bad
arguments are rejected before anything is enqueued (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(cp_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol():
    names = _declared_functions()
    assert "cp_kv_append" in names and "cp_prefill_chunk_attn" in names and "cp_mixed_step" in names
    assert "cp_prefill_chunk" in names
    L = ctypes.CDLL(cp.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert cp.cp_abi_version() == 1


def test_chunk_plan_matches_oracle():
    for n in list(range(0, 300, 7)) + [1000, 1137, 1200, 4000, 20000]:
        for W in (1, 3, 64, 256, 512):
            assert cp.cp_chunk_plan(n, W) == oracle.chunk_plan(n, W), (n, W)


def test_ladder_matches_oracle():
    for W in range(1, 2049):
        assert cp.cp_query_ladder(W) == oracle.query_ladder(W), W
    for W in (1, 2, 7, 512, 1000):
        for r in range(1, W + 1):
            assert cp.cp_query_width(r, W) == oracle.query_width(r, W)
    with pytest.raises(cp.CPError):
        cp.cp_query_width(513, 512)


def test_aligned_length_matches_oracle():
    for n in range(0, 3000, 17):
        for c in (1, 64, 256):
            assert cp.cp_aligned_length(n, c) == oracle.left_pad_length(n, c)


def test_rolling_mask_matches_oracle():
    for c, C, lp, L in [(256, 1024, 48, 2048), (256, 1024, 68, 768), (2, 8, 0, 8), (4, 4, 3, 12), (5, 8, 2, 15)]:
        for k in range(L // c):
            got = cp.cp_rolling_mask(c, C, k, lp).numpy()
            want = oracle.rolling_mask(c, C, k, lp)
            assert np.array_equal(got, want.astype(np.float32)), (c, C, lp, k)


def _flatten(steps):
    out = []
    for si, (dec, chunks) in enumerate(steps):
        out += [(si, s, -1, 1) for s in dec]
        out += [(si, s, st, r) for s, st, r in chunks]
    return out


def test_schedule_matches_oracle():
    for budget, nrun, prompts in [(8192, 64, [20000] * 4), (2048, 64, [20000] * 4), (10, 3, [9, 4]),
                                  (37, 5, [100, 3, 50, 1]), (300, 0, [1000, 999]), (5, 2, [])]:
        assert cp.cp_schedule(budget, nrun, prompts) == _flatten(oracle.schedule(budget, nrun, prompts))
    with pytest.raises(cp.CPError):
        cp.cp_schedule(4, 4, [10])


def _desc(**kw):
    base = dict(dtype=torch.bfloat16, batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                kind=cp.CP_CACHE_CONTIG, capacity=8192)
    base.update(kw)
    return cp.layer_desc(**base)


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (checks fail first)


def _prefill(desc, rows=512, real=512, max_past=0, q=FAKE, out=FAKE, lens=FAKE, ws=None):
    L = cp.lib()
    return L.cp_prefill_chunk_attn(ctypes.byref(desc), q, FAKE, FAKE, lens, None, None, rows, real,
                                   max_past, out, ws, 0, 1, None, None)


def test_prefill_rejects_bad_arguments_before_launch():
    assert _prefill(_desc(head_dim=96)) == cp.CP_ERR_UNSUPPORTED
    assert _prefill(_desc(num_q_heads=30)) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(), rows=100, real=101) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(), max_past=8192 - 511) == cp.CP_ERR_CAPACITY
    assert _prefill(_desc(), q=FAKE + 8) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(), q=None) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(dtype=7)) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(kind=cp.CP_CACHE_ROLLING, capacity=1024), rows=256, real=200) == cp.CP_ERR_INVALID_ARG
    assert _prefill(_desc(kind=cp.CP_CACHE_ROLLING, capacity=128), rows=256, real=256) == cp.CP_ERR_CAPACITY
    assert _prefill(_desc(kind=cp.CP_CACHE_PAGED, page_size=24, num_pages=8, max_blocks=4)) == cp.CP_ERR_UNSUPPORTED
    # Decode rows need the split-KV workspace.
    assert _prefill(_desc(), rows=1, real=1, max_past=100, ws=None) == cp.CP_ERR_WORKSPACE


def _chunk(desc, rows=512, real=512, max_past=0, k_new=FAKE, ws=FAKE, ws_bytes=1 << 30):
    L = cp.lib()
    return L.cp_prefill_chunk(ctypes.byref(desc), FAKE, k_new, FAKE, FAKE, FAKE, FAKE, None, None, rows, real,
                              max_past, FAKE, ws, ws_bytes, None, None)


def test_fused_chunk_rejects_bad_arguments_before_launch():
    assert _chunk(_desc(head_dim=96)) == cp.CP_ERR_UNSUPPORTED
    # a GQA group the tensor-core kernel does not take is refused before the append is enqueued
    assert _chunk(_desc(num_q_heads=32, num_kv_heads=1)) == cp.CP_ERR_UNSUPPORTED
    assert _chunk(_desc(num_q_heads=24, num_kv_heads=8)) == cp.CP_ERR_UNSUPPORTED
    assert _chunk(_desc(), rows=100, real=101) == cp.CP_ERR_INVALID_ARG
    assert _chunk(_desc(), max_past=8192 - 511) == cp.CP_ERR_CAPACITY
    assert _chunk(_desc(), k_new=None) == cp.CP_ERR_INVALID_ARG
    assert _chunk(_desc(), k_new=FAKE + 8) == cp.CP_ERR_INVALID_ARG
    # the copy of the lengths always needs the workspace; one-row chunks (decode) need the partials too
    assert _chunk(_desc(), ws=None) == cp.CP_ERR_WORKSPACE
    assert _chunk(_desc(), ws_bytes=511) == cp.CP_ERR_WORKSPACE
    need = 256 + 256 + 32 * 1 * 130 * 4  # control block, lengths copy, one row's split partials
    assert _chunk(_desc(), rows=1, real=1, max_past=100, ws_bytes=need - 1) == cp.CP_ERR_WORKSPACE
    assert _chunk(_desc(), ws=FAKE + 4) == cp.CP_ERR_WORKSPACE
    # the same layout rules as the separate calls
    assert _chunk(_desc(kind=cp.CP_CACHE_ROLLING, capacity=1024), rows=256, real=200) == cp.CP_ERR_INVALID_ARG
    assert _chunk(_desc(kind=cp.CP_CACHE_ROLLING, capacity=128), rows=256, real=256) == cp.CP_ERR_CAPACITY
    assert _chunk(_desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)) == cp.CP_ERR_INVALID_ARG


def test_append_and_mixed_reject_bad_arguments():
    L = cp.lib()
    d = _desc()
    assert L.cp_kv_append(ctypes.byref(d), FAKE, FAKE, 16, FAKE, FAKE, FAKE, None, 8190, None, None) == cp.CP_ERR_CAPACITY
    assert L.cp_kv_append(ctypes.byref(d), FAKE, None, 16, FAKE, FAKE, FAKE, None, 0, None, None) == cp.CP_ERR_INVALID_ARG
    pd = _desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)
    assert L.cp_kv_append(ctypes.byref(pd), FAKE, FAKE, 16, FAKE, FAKE, FAKE, None, 0, None, None) == cp.CP_ERR_INVALID_ARG
    # mixed step: contiguous layout unsupported, max_ctx beyond the block table rejected
    assert L.cp_mixed_step(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, FAKE, 1 << 20, None, None) == cp.CP_ERR_UNSUPPORTED
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 8 * 16 + 1,
                           FAKE, FAKE, 1 << 20, None, None) == cp.CP_ERR_CAPACITY
    # refused before the append is enqueued: a group the tensor-core kernel does not take, and a
    # workspace too small for the split-KV partials (a launch here, without a GPU, would give CP_ERR_CUDA)
    pg = _desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8, num_q_heads=32, num_kv_heads=1)
    assert L.cp_mixed_step(ctypes.byref(pg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, FAKE, 1 << 20, None, None) == cp.CP_ERR_UNSUPPORTED
    # a mixed step puts one row per sequence on the split-KV path: 2 rows of partials here
    need = 2 * 32 * 1 * (128 + 2) * 4
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, None, 0, None, None) == cp.CP_ERR_WORKSPACE
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, FAKE, need - 16, None, None) == cp.CP_ERR_WORKSPACE


def test_varlen_rejects_bad_arguments():
    """cp_prefill_varlen: contiguous caches only, at most desc->batch sequences,
    max_ctx within the capacity, 16-byte alignment, a workspace for the
    decode rows' partials; all refused before anything is enqueued."""
    L = cp.lib()
    d = _desc(batch=4)

    def call(desc=d, num_seqs=2, total=10, max_ctx=100, q=FAKE, ws=FAKE, ws_bytes=1 << 20):
        return L.cp_prefill_varlen(ctypes.byref(desc), q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, num_seqs, total,
                                   max_ctx, FAKE, ws, ws_bytes, None, None)

    pd = _desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)
    assert call(desc=pd) == cp.CP_ERR_UNSUPPORTED
    assert call(desc=_desc(kind=cp.CP_CACHE_ROLLING, capacity=1024)) == cp.CP_ERR_UNSUPPORTED
    assert call(num_seqs=5) == cp.CP_ERR_INVALID_ARG
    assert call(num_seqs=0) == cp.CP_ERR_INVALID_ARG
    assert call(max_ctx=8193) == cp.CP_ERR_CAPACITY
    assert call(q=FAKE + 8) == cp.CP_ERR_INVALID_ARG
    assert call(q=None) == cp.CP_ERR_INVALID_ARG
    assert call(ws=None, ws_bytes=0) == cp.CP_ERR_WORKSPACE
    assert call(ws=FAKE + 4) == cp.CP_ERR_WORKSPACE
    assert call(desc=_desc(batch=4, num_q_heads=32, num_kv_heads=1)) == cp.CP_ERR_UNSUPPORTED
    assert call(total=0) == cp.CP_OK  # nothing to do


def _order(max_rows, num_seqs, ppt=64):
    """The ragged calls' work list: one 8-byte entry per pair of ppt tokens
    (2 * 128 / G; G = 4 here), one more per sequence, plus 16 bytes of alignment."""
    return (-(-max_rows // ppt) + num_seqs) * 8 + 16


def test_workspace_size_formula():
    d = _desc()
    # split-KV partials for up to min(rows per sequence, 16 / G) rows per sequence (G = 4 here)
    assert cp.cp_workspace_size(d, 8, 1, 2) == 256 + 256 + 2 * 4 * 32 * 1 * 130 * 4 + _order(8, 2)
    assert cp.cp_workspace_size(d, 4, 1, 2) == 256 + 256 + 2 * 2 * 32 * 1 * 130 * 4 + _order(4, 2)
    assert cp.cp_workspace_size(d, 512, 1, 1) == 256 + 256 + 4 * 32 * 1 * 130 * 4 + _order(512, 1)
    # a 256-byte control block, a copy of the lengths in 256-byte blocks, then
    # num_seqs * Hq * ceil(ctx / 512) * (D + 2) floats of split partials, then
    # the work list
    assert cp.cp_workspace_size(d, 64, 8192, 64) == 256 + 256 + 64 * 32 * 16 * 130 * 4 + _order(64, 64)
    assert cp.cp_workspace_size(d, 1, 1, 1) == 256 + 256 + 32 * 1 * 130 * 4 + _order(1, 1)
    assert cp.cp_workspace_size(d, 1, 1, 65) == 256 + 512 + 65 * 32 * 1 * 130 * 4 + _order(1, 65)
    # fp32 layers run no tensor-core kernel: no work list
    assert cp.cp_workspace_size(_desc(dtype=torch.float32), 1, 1, 1) == 256 + 256 + 32 * 1 * 130 * 4


def test_mixed_step_rejects_misaligned_workspace():
    """The decode rows' float partials need a 16-byte aligned workspace; a
    misaligned one is refused before the append is enqueued."""
    L = cp.lib()
    pd = _desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, FAKE + 4, 1 << 20, None, None) == cp.CP_ERR_WORKSPACE


def _mixed_pair(desc, num_seqs=2, total_rows=10, max_ctx=100, q=FAKE, out=FAKE):
    """Status of cp_mixed_step (with an ample aligned workspace) and of
    cp_mixed_step_noalloc on the same arguments."""
    L = cp.lib()
    a = L.cp_mixed_step(ctypes.byref(desc) if desc is not None else None, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                        FAKE, num_seqs, total_rows, max_ctx, out, FAKE, 1 << 30, None, None)
    b = L.cp_mixed_step_noalloc(ctypes.byref(desc) if desc is not None else None, q, FAKE, FAKE, FAKE, FAKE, FAKE,
                                FAKE, FAKE, num_seqs, total_rows, max_ctx, out, None, None)
    return a, b


def test_noalloc_status_codes_match_mixed_step():
    """cp_mixed_step_noalloc makes the same argument checks as cp_mixed_step, in
    the same order, and returns the same status for each bad argument."""
    pd = dict(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)
    cases = [
        (_desc(head_dim=96, **pd), {}, cp.CP_ERR_UNSUPPORTED),
        (_desc(kind=cp.CP_CACHE_PAGED, page_size=24, num_pages=64, max_blocks=8), {}, cp.CP_ERR_UNSUPPORTED),
        (_desc(), {}, cp.CP_ERR_UNSUPPORTED),                                  # contiguous layout
        (_desc(num_q_heads=30, **pd), {}, cp.CP_ERR_INVALID_ARG),              # Hq % Hkv != 0
        (_desc(num_q_heads=32, num_kv_heads=1, **pd), {}, cp.CP_ERR_UNSUPPORTED),  # group 32
        (_desc(dtype=7, **pd), {}, cp.CP_ERR_INVALID_ARG),
        (_desc(**pd), dict(num_seqs=0), cp.CP_ERR_INVALID_ARG),
        (_desc(**pd), dict(total_rows=-1), cp.CP_ERR_INVALID_ARG),
        (_desc(**pd), dict(q=None), cp.CP_ERR_INVALID_ARG),
        (_desc(**pd), dict(out=FAKE + 8), cp.CP_ERR_INVALID_ARG),
        (_desc(**pd), dict(max_ctx=8 * 16 + 1), cp.CP_ERR_CAPACITY),
        (_desc(**pd), dict(total_rows=0), cp.CP_OK),                           # nothing to do
        (None, {}, cp.CP_ERR_INVALID_ARG),
    ]
    for desc, kw, want in cases:
        a, b = _mixed_pair(desc, **kw)
        assert a == want and b == want, (kw, a, b, want)


def test_overlap_status_codes_match_mixed_step():
    """cp_mixed_step_overlap makes cp_mixed_step's argument checks first and
    returns the same status; then it refuses a missing side stream or event and
    a side stream equal to the main one (handles here are never used: every
    case stops before anything is enqueued)."""
    L = cp.lib()
    pd = dict(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=64, max_blocks=8)
    SIDE, EV1, EV2 = 0x2000, 0x3000, 0x4000

    def ov(desc, num_seqs=2, total_rows=10, max_ctx=100, q=FAKE, out=FAKE, stream=None, side=SIDE, ev1=EV1,
           ev2=EV2):
        return L.cp_mixed_step_overlap(ctypes.byref(desc) if desc is not None else None, q, FAKE, FAKE, FAKE, FAKE,
                                       FAKE, FAKE, FAKE, num_seqs, total_rows, max_ctx, out, FAKE, 1 << 30, None,
                                       stream, side, ev1, ev2)

    for desc, kw in [(_desc(head_dim=96, **pd), {}), (_desc(), {}), (_desc(num_q_heads=30, **pd), {}),
                     (_desc(**pd), dict(num_seqs=0)), (_desc(**pd), dict(q=None)),
                     (_desc(**pd), dict(max_ctx=8 * 16 + 1)), (None, {})]:
        want, _ = _mixed_pair(desc, **kw)
        assert want != cp.CP_OK and ov(desc, **kw) == want, kw
    d = _desc(**pd)
    assert ov(d, total_rows=0) == cp.CP_OK
    assert ov(d, side=None) == cp.CP_ERR_INVALID_ARG
    assert ov(d, ev1=None) == cp.CP_ERR_INVALID_ARG
    assert ov(d, ev2=None) == cp.CP_ERR_INVALID_ARG
    assert ov(d, stream=SIDE) == cp.CP_ERR_INVALID_ARG


def test_noalloc_refuses_a_step_whose_partials_exceed_the_scratch():
    """The fixed scratch is compared with the split-KV partials cp_mixed_step
    would use for the step: one sequence more than fits is refused with
    CP_ERR_WORKSPACE before anything is enqueued."""
    L = cp.lib()
    d = _desc(kind=cp.CP_CACHE_PAGED, page_size=16, num_pages=1 << 20, max_blocks=1 << 12)
    per_seq = 32 * ((8192 + 511) // 512) * (128 + 2) * 4     # partials of one sequence at max_ctx 8192
    fits = cp.cp_noalloc_scratch_bytes() // per_seq           # sequences whose partials fit the array
    st = L.cp_mixed_step_noalloc(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, fits + 1,
                                 fits + 1, 8192, FAKE, None, None)
    assert st == cp.CP_ERR_WORKSPACE


def test_selftest_rejects_bad_pointers_before_launch():
    """The bounded-wait self-test checks its pointers on the host (no launch)."""
    L = cp.lib()
    f = L.cp_selftest_bounded_wait
    assert f(None, None, None) == cp.CP_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(16), None, None) == cp.CP_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(16), ctypes.c_void_p(20), None) == cp.CP_ERR_INVALID_ARG  # not 8-byte aligned


def test_every_bound_entry_point_declares_its_argument_types():
    """Every C function the binding calls has ctypes argtypes, so no 64-bit
    pointer or stream handle is passed as a 32-bit int."""
    import re
    src = open(cp.__file__).read()
    called = set(re.findall(r"lib\(\)\.(cp_\w+)\(", src))
    L = cp.lib()
    missing = [name for name in sorted(called) if getattr(L, name).argtypes is None]
    assert not missing, missing


def test_varlen_overlap_status_codes_match_varlen():
    """cp_prefill_varlen_overlap makes cp_prefill_varlen's checks first, with
    the same status codes, then refuses a missing side stream or event and a
    side stream equal to the main one (no case enqueues anything)."""
    L = cp.lib()
    SIDE, EV1, EV2 = 0x2000, 0x3000, 0x4000

    def both(desc, num_seqs=2, total_rows=10, max_ctx=100, q=FAKE, ws=FAKE, ws_bytes=1 << 30):
        d = ctypes.byref(desc) if desc is not None else None
        plain = L.cp_prefill_varlen(d, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, num_seqs, total_rows, max_ctx, FAKE,
                                    ws, ws_bytes, None, None)
        over = L.cp_prefill_varlen_overlap(d, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, num_seqs, total_rows, max_ctx,
                                           FAKE, ws, ws_bytes, None, None, SIDE, EV1, EV2)
        return plain, over

    cases = [(_desc(batch=4, head_dim=96), {}), (_desc(batch=4, kind=cp.CP_CACHE_PAGED, page_size=16,
                                                     num_pages=8, max_blocks=4), {}),
             (_desc(batch=4, num_q_heads=30), {}), (_desc(batch=4), dict(num_seqs=5)),
             (_desc(batch=4), dict(q=None)), (_desc(batch=4), dict(q=FAKE + 8)),
             (_desc(batch=4), dict(max_ctx=8193)), (_desc(batch=4), dict(ws=None)), (None, {})]
    for desc, kw in cases:
        plain, over = both(desc, **kw)
        assert plain != cp.CP_OK and over == plain, (kw, plain, over)
    d = _desc(batch=4)
    assert both(d, total_rows=0) == (cp.CP_OK, cp.CP_OK)

    def ov(**kw):
        a = dict(side=SIDE, ev1=EV1, ev2=EV2, stream=None)
        a.update(kw)
        return L.cp_prefill_varlen_overlap(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                                           FAKE, FAKE, 1 << 30, None, a["stream"], a["side"], a["ev1"], a["ev2"])
    assert ov(side=None) == cp.CP_ERR_INVALID_ARG
    assert ov(ev1=None) == cp.CP_ERR_INVALID_ARG
    assert ov(ev2=None) == cp.CP_ERR_INVALID_ARG
    assert ov(stream=SIDE) == cp.CP_ERR_INVALID_ARG
