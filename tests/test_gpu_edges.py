"""GPU parity at the edges of the sizes the contiguous path accepts: a cache
filled to exactly its physical capacity (capacities that are not a multiple of
the 128-key tile), the widest chunk (a 4000-token prompt in one call), and the
largest query-head group, each through the one-call chunk entry point and
through the separate append + attention calls."""
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


def _both_paths(n, W, hq, hkv, d, dtype, cap, seed):
    q, k, v = SI.gqa_prompt(n, seed=seed, hq=hq, hkv=hkv, dim=d, dtype=dtype)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    fused = Contig(dtype, hq, hkv, d, cap=cap, fused=True)
    split = Contig(dtype, hq, hkv, d, cap=cap)
    out_f, _ = prefill(fused, qd, kd, vd, W)
    out_s, _ = prefill(split, qd, kd, vd, W)
    torch.cuda.synchronize()
    for c in (fused, split):
        assert int(c.lens.item()) == n and int(c.status.item()) == 0
        assert torch.equal(c.k[0, :, :n].cpu(), k.permute(1, 0, 2))
        assert torch.equal(c.v[0, :, :n].cpu(), v.permute(1, 0, 2))
        if n < cap:
            assert torch.isnan(c.k[0, :, n:].float()).all() and torch.isnan(c.v[0, :, n:].float()).all()
    assert torch.equal(out_f, out_s)
    return q, k, v, out_f


@pytest.mark.parametrize("n,W,hq,hkv,d,dtype", [
    (700, 256, 32, 8, 128, torch.bfloat16),   # 256 + 256 + 188: the last chunk ends at slot 699
    (389, 128, 16, 2, 128, torch.float16),    # GQA 8, capacity 389
    (530, 200, 8, 2, 64, torch.bfloat16),     # head_dim 64, capacity 530
    (257, 257, 16, 1, 64, torch.float16),     # GQA 16 (one KV head), one chunk filling the cache
    (129, 64, 4, 4, 128, torch.bfloat16),     # MHA, capacity one past a tile
])
def test_cache_filled_to_capacity(n, W, hq, hkv, d, dtype):
    """Cache capacity == prompt length: the last chunk writes the last slot
    and its key walk ends exactly at the capacity."""
    q, k, v, out = _both_paths(n, W, hq, hkv, d, dtype, cap=n, seed=n + 7)
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    err = np.abs(f64(out) - ref).max()
    assert err < BF16_TOL, err


def test_fp32_cache_filled_to_capacity():
    """The fp32 path with capacity == prompt length (300 tokens, chunks of
    128, 8 heads x 64): every element against the oracle at 1e-4."""
    n, W = 300, 128
    q, k, v, out = _both_paths(n, W, 8, 8, 64, torch.float32, cap=n, seed=5)
    ref, _, _ = oracle.chunked_prefill(f64(q), f64(k), f64(v), W)
    assert np.abs(f64(out) - ref).max() < F32_TOL


def test_widest_chunk_one_call():
    """The 4000-token GQA 32/8 x 128 bf16 prompt as one chunk of 4000 rows (a
    chunk width of 4096) into a cache of capacity 4000: sampled rows against
    the oracle one by one, the cache byte for byte, the two paths bit for bit."""
    n = 4000
    assert cp.cp_chunk_plan(n, 4096) == [n]
    q, k, v, out = _both_paths(n, 4096, 32, 8, 128, torch.bfloat16, cap=n, seed=1)
    rng = np.random.default_rng(4)
    rows = [0, 1, 127, 128, 2047, n - 2, n - 1] + list(rng.integers(0, n, 25))
    kk, vv, qq, oo = f64(k), f64(v), f64(q), f64(out)
    worst = max(np.abs(oo[p] - oracle.attention_row(qq[p], kk, vv, int(p))).max() for p in rows)
    assert worst < BF16_TOL, worst
    assert np.isfinite(oo).all()
