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
    assert _chunk(_desc(), ws_bytes=255) == cp.CP_ERR_WORKSPACE
    need = cp.cp_workspace_size(_desc(), 1, 101, 1)
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
    need = cp.cp_workspace_size(pd, 10, 100, 2)
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, None, 0, None, None) == cp.CP_ERR_WORKSPACE
    assert L.cp_mixed_step(ctypes.byref(pd), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 100,
                           FAKE, FAKE, need // 4, None, None) == cp.CP_ERR_WORKSPACE


def test_workspace_size_formula():
    d = _desc()
    # a copy of the lengths in 256-byte blocks, then num_seqs * Hq * ceil(ctx / 512) * (D + 2)
    # floats of split partials
    assert cp.cp_workspace_size(d, 64, 8192, 64) == 256 + 64 * 32 * 16 * 130 * 4
    assert cp.cp_workspace_size(d, 1, 1, 1) == 256 + 32 * 1 * 130 * 4
    assert cp.cp_workspace_size(d, 1, 1, 65) == 512 + 65 * 32 * 1 * 130 * 4
