"""Pins for the CPU oracle: each function checks the oracle against something
other than itself (values printed on the pages, closed forms, invariants,
brute force on tiny inputs, an independent library routine) and raises
AssertionError on a mismatch.

``test_oracle.py`` runs every pin; ``test_oracle_mutants.py`` plants plausible
mistakes in the oracle and checks that at least one pin catches each of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle.cp_oracle as O
import synth_inputs as SI

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------- plans

def pin_chunk_plan_printed():
    """Chunk sizes printed on the pages (glossary example; wiki section 三)."""
    for case in _golden("chunk_plans.json")["cases"]:
        assert O.chunk_plan(case["n"], case["W"]) == case["sizes"], case


def pin_chunk_plan_invariants():
    """Sizes sum to n, all but the last equal W, the last is in [1, W]."""
    for n in range(0, 700, 7):
        for W in (1, 3, 64, 100, 256, 512):
            s = O.chunk_plan(n, W)
            assert sum(s) == n
            assert len(s) == -(-n // W)
            assert all(x == W for x in s[:-1])
            if s:
                assert 1 <= s[-1] <= W


def pin_ladder_printed():
    """{171, 342, 512} for W = 512, at most 170 wasted rows, 311 rows -> 342
    where a power-of-two ladder would give 512 (about 65% more)."""
    g = _golden("query_ladder.json")
    assert O.query_ladder(g["W"]) == g["tiers"]
    waste = max(O.query_width(r, g["W"]) - r for r in range(1, g["W"] + 1))
    assert waste == g["max_waste_rows"]
    w = O.query_width(g["pow2_rows"], g["W"])
    assert w == 342
    pow2 = 1 << (g["pow2_rows"] - 1).bit_length()
    assert pow2 == g["pow2_width"]
    assert round(100 * (pow2 - g["pow2_rows"]) / g["pow2_rows"]) == g["pow2_extra_percent"]


def pin_ladder_invariants():
    """The top tier equals W for every width 1..4096, there are at most three
    tiers, they are increasing, and every r in 1..W maps to the smallest tier >= r."""
    for W in range(1, 4097):
        t = O.query_ladder(W)
        assert t[-1] == W, W
        assert 1 <= len(t) <= 3
        assert all(a < b for a, b in zip(t, t[1:]))
    for W in (1, 2, 5, 100, 512, 1000):
        t = O.query_ladder(W)
        for r in range(1, W + 1):
            w = O.query_width(r, W)
            assert w >= r and w in t
            assert all(x < r for x in t if x < w)


def pin_schedule_hand_example():
    """Budget 10, three running decodes, prompts of 9 and 4 tokens, worked by
    hand from the glossary's rule: decodes first, then waiting prompt chunks;
    an unfinished prompt continues next step; a finished one decodes after."""
    steps = O.schedule(10, 3, [9, 4])
    assert steps == [
        ([0, 1, 2], [(3, 0, 7)]),
        ([0, 1, 2], [(3, 7, 2), (4, 0, 4)]),
    ], steps
    steps = O.schedule(6, 1, [3, 3, 3])
    assert steps == [
        ([0], [(1, 0, 3), (2, 0, 2)]),
        ([0, 1], [(2, 2, 1), (3, 0, 3)]),
    ], steps


def pin_schedule_invariants():
    """Every step fits the budget, each prompt's tokens are scheduled once, in
    order, and the decode set only grows by prompts that just finished."""
    for budget, nrun, prompts in [(8192, 64, [20000] * 4), (2048, 64, [20000] * 4),
                                  (37, 5, [100, 3, 50, 1]), (300, 0, [1000, 999])]:
        steps = O.schedule(budget, nrun, prompts)
        pos = [0] * len(prompts)
        dec = list(range(nrun))
        for d, chunks in steps:
            assert d == dec
            assert len(d) + sum(r for _, _, r in chunks) <= budget
            fin = []
            for sid, start, r in chunks:
                i = sid - nrun
                assert start == pos[i] and r >= 1
                pos[i] += r
                if pos[i] == prompts[i]:
                    fin.append(sid)
            dec = dec + fin
        assert pos == prompts
    # The 8192 / 2048 budgets over 64 decodes and four 20000-token prompts.
    s8 = O.schedule(8192, 64, [20000] * 4)
    assert len(s8) == 10
    assert s8[0][1] == [(64, 0, 8128)]
    assert s8[2][1] == [(64, 16256, 3744), (65, 0, 4384)]
    assert len(O.schedule(2048, 64, [20000] * 4)) == 41


# ----------------------------------------------------------------- attention

def _brute_attention(q, k, v, vis, scale):
    """Pure-Python loops: softmax-weighted average of visible value rows."""
    n, d = len(q), len(q[0])
    out = []
    for i in range(n):
        s = [scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in range(len(k)) if vis(i, j)]
        idx = [j for j in range(len(k)) if vis(i, j)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        z = sum(w)
        out.append([sum(w[a] * v[idx[a]][t] for a in range(len(idx))) / z for t in range(d)])
    return out


def pin_brute_force_tiny():
    """Oracle one-shot, chunked and single-chunk attention equal pure-Python
    loops on tiny GQA shapes (2 KV heads, 4 query heads)."""
    rng = _rng(1)
    n, hq, hkv, d = 7, 4, 2, 3
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    scale = 1.0 / math.sqrt(d)
    want = np.empty((n, hq, d))
    for h in range(hq):
        g = h // 2
        want[:, h] = _brute_attention(q[:, h].tolist(), k[:, g].tolist(), v[:, g].tolist(),
                                      lambda i, j: j <= i, scale)
    got = O.causal_attention(q, k, v)
    assert np.allclose(got, want, rtol=0, atol=1e-12)
    out, _, _ = O.chunked_prefill(q, k, v, 3)
    assert np.allclose(out, want, rtol=0, atol=1e-12)
    # Rows 4..6 as one chunk over a cache of positions 0..6.
    got = O.chunk_attention(q[4:7], k, v, 4)
    assert np.allclose(got, want[4:7], rtol=0, atol=1e-12)


def pin_value_ones():
    """V = 1 everywhere gives O = 1 everywhere (softmax weights sum to one)."""
    rng = _rng(2)
    q = rng.standard_normal((20, 4, 8))
    k = rng.standard_normal((20, 2, 8))
    v = np.ones((20, 2, 8))
    out, _, _ = O.chunked_prefill(q, k, v, 6)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-13)


def pin_identity_values():
    """With V = identity (keys <= head_dim), O row i is the attention
    distribution of query i: it sums to 1, is exactly 0 past the causal edge,
    positive on [0, i], and matches softmax of the visible scores."""
    rng = _rng(3)
    n, d = 10, 16
    q = rng.standard_normal((n, 2, d))
    k = rng.standard_normal((n, 1, d))
    v = np.zeros((n, 1, d))
    v[np.arange(n), 0, np.arange(n)] = 1.0
    out, _, _ = O.chunked_prefill(q, k, v, 4)
    for h in range(2):
        p = out[:, h, :n]
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-13)
        assert np.all(p[np.triu_indices(n, 1)] == 0.0)
        assert np.all(p[np.tril_indices(n)] > 0.0)
        s = (q[:, h] @ k[:, 0].T) / math.sqrt(d)
        for i in range(n):
            e = np.exp(s[i, :i + 1] - s[i, :i + 1].max())
            assert np.allclose(p[i, :i + 1], e / e.sum(), atol=1e-13)


def pin_equal_keys_mean():
    """Identical keys give uniform weights: O row i is the mean of V rows 0..i."""
    rng = _rng(4)
    n, d = 12, 8
    q = rng.standard_normal((n, 3, d))
    k = np.repeat(rng.standard_normal((1, 1, d)), n, axis=0)
    v = rng.standard_normal((n, 1, d))
    out, _, _ = O.chunked_prefill(q, k, v, 5)
    want = np.cumsum(v[:, 0], axis=0) / np.arange(1, n + 1)[:, None]
    for h in range(3):
        assert np.allclose(out[:, h], want, atol=1e-13)


def pin_dominant_key():
    """A query aligned with one visible key, scaled up, puts all its weight on
    that key: O equals that key's V row (to within exp(-large))."""
    n, d = 6, 8
    k = np.zeros((n, 1, d))
    k[np.arange(n), 0, np.arange(n)] = 1.0  # orthonormal keys
    v = _rng(5).standard_normal((n, 1, d))
    q = np.zeros((n, 1, d))
    target = [0, 0, 1, 3, 2, 5]  # each target <= row index
    for i, j in enumerate(target):
        q[i, 0, j] = 400.0
    out = O.causal_attention(q, k, v)
    assert np.allclose(out[:, 0], v[target, 0], atol=1e-12)


def pin_torch_sdpa_example():
    """The glossary's one-layer example: 1000 tokens, chunks of 256, 8 heads x 64,
    drawn with seed 0.  The oracle's chunked output matches torch's one-shot
    causal attention (an independent implementation) within the printed
    tolerance 1e-5, in four chunks."""
    g = _golden("sdpa_example.json")
    q, k, v = SI.fp32_sdpa_example(g["seed"], g["prompt_len"], g["heads"], g["head_dim"])
    full = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None],
        is_causal=True)[0].permute(1, 0, 2).numpy()
    out, _, sizes = O.chunked_prefill(q.numpy(), k.numpy(), v.numpy(), g["chunk"])
    assert len(sizes) == g["n_chunks"]
    assert bool(np.allclose(full, out, rtol=0, atol=g["atol"])) == g["same_result"]


def pin_chunked_equals_one_shot():
    """Chunking changes only the order of the work ([Wiki] 一.2): the chunked
    output equals one-shot causal attention for several chunk widths."""
    rng = _rng(6)
    n, d = 37, 16
    q = rng.standard_normal((n, 8, d))
    k = rng.standard_normal((n, 2, d))
    v = rng.standard_normal((n, 2, d))
    ref = O.causal_attention(q, k, v)
    for W in (1, 5, 16, 36, 37, 64):
        out, _, _ = O.chunked_prefill(q, k, v, W)
        assert np.allclose(out, ref, rtol=0, atol=1e-12), W


def pin_cache_prefix_bytes():
    """After chunk k the cache equals the same-length prefix of the cache a
    one-shot pass writes, byte for byte, and slots past it are untouched
    ([Wiki] 一.1)."""
    rng = _rng(7)
    n, d, cap = 23, 8, 40
    q = rng.standard_normal((n, 4, d)).astype(np.float32)
    k = rng.standard_normal((n, 2, d)).astype(np.float32)
    v = rng.standard_normal((n, 2, d)).astype(np.float32)
    one_k = O.kv_append(O.new_cache(1, 2, cap, d), k[None], [0])
    _, snaps, sizes = O.chunked_prefill(q, k, v, 6, capacity=cap)
    end = 0
    for (kc, vc), r in zip(snaps, sizes):
        end += r
        assert kc.tobytes() == np.concatenate(
            [one_k[:, :, :end], np.zeros((1, 2, cap - end, d), np.float32)], axis=2).tobytes()
        assert np.array_equal(vc[0, :, :end], np.transpose(v[:end], (1, 0, 2)))


def pin_gqa_is_repeated_mha():
    """A GQA layer equals multi-head attention whose K/V heads are each
    repeated Hq/Hkv times in order (contiguous groups)."""
    rng = _rng(8)
    n, d = 15, 8
    q = rng.standard_normal((n, 8, d))
    k = rng.standard_normal((n, 2, d))
    v = rng.standard_normal((n, 2, d))
    mha = O.causal_attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1))
    out, _, _ = O.chunked_prefill(q, k, v, 4)
    assert np.allclose(out, mha, atol=1e-13)
    # Different KV heads must give different outputs for the two groups.
    assert not np.allclose(out[:, 0], O.causal_attention(q[:, :1], k[:, 1:], v[:, 1:])[:, 0])


def pin_padding_invisible():
    """Padding a chunk by repeating its last row leaves the real rows' outputs
    unchanged, writes the pad rows' K/V after the real ones, and rewinds the
    valid length to past + real rows ([Wiki] 四)."""
    rng = _rng(9)
    n, d, W, cap = 29, 8, 12, 64
    q = rng.standard_normal((n, 4, d))
    k = rng.standard_normal((n, 2, d))
    v = rng.standard_normal((n, 2, d))
    ref = O.causal_attention(q, k, v)
    kc = O.new_cache(1, 2, cap, d, np.float64)
    vc = O.new_cache(1, 2, cap, d, np.float64)
    past = 0
    for r in O.chunk_plan(n, W):
        out, kc, vc, new_past, rp = O.padded_chunk(q[past:past + r], k[past:past + r],
                                                   v[past:past + r], kc, vc, past, W)
        assert rp == O.query_width(r, W) and rp >= r
        assert np.allclose(out, ref[past:past + r], atol=1e-12)
        for t in range(r, rp):  # pad slots hold copies of the last real row
            assert np.array_equal(kc[0, :, past + t], k[past + r - 1])
        assert new_past == past + r
        past = new_past
    assert past == n


def pin_rolling_mask_examples():
    """Hand-worked masks.  c=2, C=8, chunk 0, no pad: slots 6 and 7 hold
    positions 0 and 1, so row 0 may see slot 6 and row 1 slots 6-7; the allowed
    entries sit at the right end and the rest is filled with -32768 ([Horizon] 4)."""
    m = O.rolling_mask(2, 8, 0, 0)
    assert m.shape == (2, 8)
    want = np.full((2, 8), -32768.0)
    want[0, 6] = 0.0
    want[1, 6:] = 0.0
    assert np.array_equal(m, want)
    # C = 8 holding 5 valid tokens (c = 5, chunk 0): the valid slots are 3..7.
    m = O.rolling_mask(5, 8, 0, 0)
    assert np.all(m[:, :3] == -32768.0)
    assert np.all(m[-1, 3:] == 0.0)
    # Left pad of 3 (chunk 0 of c=4, C=4): slots holding positions < 3 are masked.
    m = O.rolling_mask(4, 4, 0, 3)
    assert np.all(m[:, :3] == -32768.0) and m[3, 3] == 0.0
    # Second chunk, C = c = 4: full window of the current chunk only.
    m = O.rolling_mask(4, 4, 1, 0)
    assert np.array_equal(m == 0.0, np.tril(np.ones((4, 4), bool)))


def pin_rolling_no_overflow_is_plain_prefill():
    """C >= L: nothing is ever dropped and chunk prefill equals ordinary causal
    prefill over the real (unpadded) tokens ([Horizon] 3)."""
    rng = _rng(10)
    n_real, c, C, d = 22, 8, 32, 8
    L = O.left_pad_length(n_real, c)
    lp = L - n_real
    q = rng.standard_normal((L, 3, d))
    k = rng.standard_normal((L, 3, d))
    v = rng.standard_normal((L, 3, d))
    out, snaps = O.rolling_prefill(q, k, v, c, C, lp)
    ref = O.causal_attention(q[lp:], k[lp:], v[lp:])
    assert np.allclose(out[lp:], ref, atol=1e-12)
    # The cache holds the newest positions at its right end.
    kc, _ = snaps[-1]
    assert np.array_equal(kc[:, C - L:], np.transpose(k, (1, 0, 2)))
    assert np.all(kc[:, :C - L] == 0.0)


def pin_rolling_sliding_window():
    """L > C: every row of chunk k attends exactly the positions
    [max(left_pad, (k+1)c - C), p] of the unrolled sequence (a sliding window
    whose oldest KV is forgotten, [Horizon] 3), computed here directly from
    index ranges instead of the rolled cache and the mask."""
    rng = _rng(11)
    n_real, c, C, d = 45, 6, 18, 4
    L = O.left_pad_length(n_real, c)
    lp = L - n_real
    q = rng.standard_normal((L, 2, d))
    k = rng.standard_normal((L, 2, d))
    v = rng.standard_normal((L, 2, d))
    out, snaps = O.rolling_prefill(q, k, v, c, C, lp)
    sc = 1.0 / math.sqrt(d)
    for p in range(lp, L):
        ci = p // c
        lo = max(lp, (ci + 1) * c - C)
        for h in range(2):
            s = sc * (k[lo:p + 1, h] @ q[p, h])
            w = np.exp(s - s.max())
            want = (w @ v[lo:p + 1, h]) / w.sum()
            assert np.allclose(out[p, h], want, atol=1e-12), (p, h)
    # After the last chunk the cache is the newest C positions, oldest first.
    kc, _ = snaps[-1]
    assert np.array_equal(kc, np.transpose(k[L - C:], (1, 0, 2)))


def pin_paged_round_trip():
    """Writing tokens through a block table and gathering them back gives the
    contiguous sequence, byte for byte, and touches only the listed pages."""
    rng = _rng(12)
    page, hkv, d, n = 4, 2, 3, 17
    table = np.array([5, 0, 3, 7, 1], np.int32)
    pool = np.full((9, hkv, page, d), np.nan)
    kv = rng.standard_normal((n, hkv, d))
    for a in range(n):
        O.paged_write(pool, table, a, kv[a])
    assert np.array_equal(O.paged_gather(pool, table, n), kv)
    for unused in (2, 4, 6, 8):
        assert np.all(np.isnan(pool[unused]))


def pin_paged_coordinates():
    """Each token lands at the (page id, slot) worked out by hand for a
    scattered block table (tests/golden/paged_layout.json), pages not in the
    table stay untouched, and the last, partly filled page has only its first
    slot written."""
    g = _golden("paged_layout.json")
    page, hkv, d = g["page"], 2, 3
    pool = np.full((g["num_pages"], hkv, page, d), np.nan)
    table = np.array(g["table"], np.int32)
    for a in range(g["n_tokens"]):
        O.paged_write(pool, table, a, np.full((hkv, d), float(a + 1)))
    for a, pid, slot in g["tokens"]:
        assert np.all(pool[pid, :, slot] == a + 1), (a, pid, slot)
    for pid in g["untouched_pages"]:
        assert np.all(np.isnan(pool[pid]))
    pf = g["partly_filled"]
    assert not np.isnan(pool[pf["page"], :, pf["written_slots"]]).any()
    assert np.isnan(pool[pf["page"], :, pf["empty_slots"]]).all()
    got = O.paged_gather(pool, table, g["n_tokens"])
    assert np.array_equal(got[:, 0, 0], np.arange(1, g["n_tokens"] + 1, dtype=np.float64))


def pin_mixed_step_composition():
    """A mixed step (decode rows + prompt chunks over pages) equals running each
    sequence's rows alone as a chunk over its own gathered cache, and the
    decode rows equal single-row attention over their whole context."""
    rng = _rng(13)
    page, hq, hkv, d = 4, 4, 2, 8
    ctx = [5, 9, 1]          # existing context of three decodes
    prompt = 11               # one prompt, first chunk of 7 rows
    rows = [1, 1, 1, 7]
    past = [ctx[0], ctx[1], ctx[2], 0]
    nseq = 4
    table = np.arange(nseq * 4, dtype=np.int32).reshape(nseq, 4)[:, ::-1].copy()
    kp = np.zeros((nseq * 4, hkv, page, d))
    vp = np.zeros((nseq * 4, hkv, page, d))
    hist_k = [rng.standard_normal((c, hkv, d)) for c in ctx] + [np.zeros((0, hkv, d))]
    hist_v = [rng.standard_normal((c, hkv, d)) for c in ctx] + [np.zeros((0, hkv, d))]
    for s in range(nseq):
        for a in range(past[s]):
            O.paged_write(kp, table[s], a, hist_k[s][a])
            O.paged_write(vp, table[s], a, hist_v[s][a])
    T = sum(rows)
    q = rng.standard_normal((T, hq, d))
    kn = rng.standard_normal((T, hkv, d))
    vn = rng.standard_normal((T, hkv, d))
    out, kp2, vp2, newp = O.mixed_step(q, kn, vn, kp, vp, table, rows, past)
    assert newp == [p + r for p, r in zip(past, rows)]
    t = 0
    for s in range(nseq):
        ks = np.concatenate([hist_k[s], kn[t:t + rows[s]]])
        vs = np.concatenate([hist_v[s], vn[t:t + rows[s]]])
        assert np.array_equal(O.paged_gather(kp2, table[s], newp[s]), ks)
        full = O.causal_attention(np.concatenate([np.zeros((past[s], hq, d)), q[t:t + rows[s]]]), ks, vs)
        assert np.allclose(out[t:t + rows[s]], full[past[s]:], atol=1e-12)
        t += rows[s]
    assert prompt > rows[-1]


ALL_PINS = [
    pin_chunk_plan_printed, pin_chunk_plan_invariants, pin_ladder_printed, pin_ladder_invariants,
    pin_schedule_hand_example, pin_schedule_invariants, pin_brute_force_tiny, pin_value_ones,
    pin_identity_values, pin_equal_keys_mean, pin_dominant_key, pin_torch_sdpa_example,
    pin_chunked_equals_one_shot, pin_cache_prefix_bytes, pin_gqa_is_repeated_mha,
    pin_padding_invisible, pin_rolling_mask_examples, pin_rolling_no_overflow_is_plain_prefill,
    pin_rolling_sliding_window, pin_paged_round_trip, pin_paged_coordinates, pin_mixed_step_composition,
]
