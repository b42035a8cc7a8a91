"""CPU oracle for chunked-prefill causal attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import, call or execute this
module.  The product path (the C-ABI library under
``chunked_prefill_causal_cp_gb300/`` and its Python binding) never imports it,
and this module imports nothing from the product path.

Plain, slow and meant to be checked by eye: numpy float64 throughout, with
numpy's matrix product as the only library primitive used as a step.  There is
no blocking, fusion or reordering beyond what the cited passages state.

Sources, cited by page title and section:

  [Wiki]      ONNX GenAI Wiki, "Chunked Prefill" (justinchuby.com).
              §一.1 KV cache is append-only; §一.2 the causal mask makes the
              split invisible; §一.3 capacity vs length (seqlens_k); §二 why
              chunk; §三 the remainder chunk; §四 query-axis padding;
              §五/§六 why three tiers, and how the step is rounded.
  [Horizon]   Horizon developer blog, "【大模型】Chunk Prefill——把一次算不动的事拆成多次".
              §2 capacity C and right alignment; §3 rolling KV cache;
              §4 per-chunk mask; §5 alignment + chunk loop; "后续" (-32768).
  [Glossary]  Ultralytics glossary, "Chunked Prefill" (zh page; the de page
              carries the same text).  "How chunked prefill works" (token
              budget scheduler and the one-layer equivalence example);
              "Related techniques" (PagedAttention).

Readings taken where the pages are silent:
  * softmax scale 1/sqrt(head_dim) (the glossary example uses the attention
    routine's default scale);
  * GQA groups are contiguous: query head h reads KV head h // (Hq / Hkv);
  * seqlens_k counts valid cache slots (= past length);
  * pad rows of a widened chunk repeat the last real row's q, k and v;
  * rolling cache starts all-zero; a slot is allowed iff it holds a real,
    already-written position at or before the query (causal and pad masks
    combined); the mask value is *added* to the scores;
  * the scheduler visits waiting prompts first-come-first-served with no
    per-prompt cap, and a prompt whose last token was scheduled decodes from
    the next step on.

Parity status: every function here is pinned by ``tests/test_oracle.py``
except the output of rows that see no key at all in rolling mode (left-pad
query rows), whose value depends on the mask constant's precision: parity
unpinned for those rows (finiteness only).
"""
from __future__ import annotations

import math

import numpy as np

# [Horizon] §4 and "后续": masked entries are filled with -32768 rather than -inf.
MASK_MIN = -32768.0


# ---------------------------------------------------------------------------
# Integer plans
# ---------------------------------------------------------------------------

def chunk_plan(n_tokens: int, W: int) -> list[int]:
    """Split a prompt of ``n_tokens`` into chunks of width ``W``.

    [Wiki] §二 (the prompt is cut with ``chunks(W)``) and §三: every chunk has W
    rows except the last, which takes the remainder.
    """
    if W <= 0 or n_tokens < 0:
        raise ValueError("W must be positive and n_tokens non-negative")
    sizes = []
    start = 0
    while start < n_tokens:
        sizes.append(min(W, n_tokens - start))
        start += W
    return sizes


def query_ladder(W: int) -> list[int]:
    """The query-width tiers for chunk width ``W``.

    [Wiki] §四: rows are rounded up to one of three evenly spaced tiers at or
    below the chunk width ({171, 342, 512} for W = 512).  [Wiki] §六: the step
    is rounded up so that the top tier lands exactly on W.  Tiers that coincide
    for tiny W are listed once.
    """
    if W <= 0:
        raise ValueError("W must be positive")
    step = -(-W // 3)  # ceil(W / 3)
    tiers: list[int] = []
    for i in (1, 2, 3):
        t = min(i * step, W)
        if t not in tiers:
            tiers.append(t)
    return tiers


def query_width(real_rows: int, W: int) -> int:
    """Smallest tier of ``query_ladder(W)`` that holds ``real_rows`` ([Wiki] §四)."""
    if not 1 <= real_rows <= W:
        raise ValueError("real_rows must be in [1, W]")
    for t in query_ladder(W):
        if t >= real_rows:
            return t
    raise AssertionError("unreachable: the top tier equals W")


def pad_rows(x: np.ndarray, rows_padded: int) -> np.ndarray:
    """Widen a per-token array ``[rows, ...]`` to ``rows_padded`` rows by repeating
    its last row ([Wiki] §四: pad rows repeat the last real token)."""
    r = x.shape[0]
    if rows_padded < r:
        raise ValueError("rows_padded < rows")
    extra = np.repeat(x[r - 1:r], rows_padded - r, axis=0)
    return np.concatenate([x, extra], axis=0)


def left_pad_length(n_real: int, c: int) -> int:
    """Aligned length: ``n_real`` rounded up to a multiple of the chunk size
    ([Horizon] §5: the alignment target is a multiple of chunk_size, so every
    chunk has the same width).  Returns the aligned length L."""
    return -(-n_real // c) * c


def schedule(budget: int, n_running: int, prompt_lens: list[int]):
    """Token-budget step plan ([Glossary] "How chunked prefill works").

    Each step first gives one token to every running decode, then fills the
    rest of the budget with chunks of waiting prompts.  A prompt that does not
    fit continues in the next step, its KV cache growing chunk by chunk; once
    its whole prompt has been processed it starts decoding (from the next
    step on).  Prompts are visited first-come-first-served.

    Sequence ids: running decodes are 0..n_running-1; prompt i is n_running+i.
    Returns a list of steps ``(decode_ids, [(seq_id, start, rows), ...])``;
    the plan ends when every prompt has been fully scheduled.
    """
    decodes = list(range(n_running))
    done = [0] * len(prompt_lens)
    steps = []
    while any(d < n for d, n in zip(done, prompt_lens)):
        left = budget - len(decodes)
        if left <= 0:
            raise ValueError("budget leaves no room for prompt tokens")
        chunks = []
        finished = []
        for i, n in enumerate(prompt_lens):
            if done[i] >= n:
                continue
            if left == 0:
                break
            take = min(left, n - done[i])
            chunks.append((n_running + i, done[i], take))
            done[i] += take
            left -= take
            if done[i] == n:
                finished.append(n_running + i)
        steps.append((list(decodes), chunks))
        decodes += finished
    return steps


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def default_scale(head_dim: int) -> float:
    """Softmax scale 1/sqrt(head_dim) (reading: the glossary example relies on
    the attention routine's default scale)."""
    return 1.0 / math.sqrt(head_dim)


def kv_head(h: int, hq: int, hkv: int) -> int:
    """KV head read by query head ``h`` (GroupQueryAttention, [Wiki] §一.3;
    reading: contiguous groups of Hq/Hkv query heads share one KV head)."""
    return h // (hq // hkv)


def causal_visible(pos_q: np.ndarray, pos_k: np.ndarray) -> np.ndarray:
    """Boolean ``[len(pos_q), len(pos_k)]``: key at absolute position a is visible
    from the query at absolute position p iff a <= p ([Wiki] §一.2; the
    glossary's mask is the lower triangle shifted by the chunk start)."""
    return pos_k[None, :] <= pos_q[:, None]


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible: np.ndarray,
           scale: float) -> np.ndarray:
    """Softmax attention of query rows over key rows with an exclusion mask.

    q ``[n, D]``, k/v ``[m, D]``, visible bool ``[n, m]`` -> ``[n, D]`` float64:
    s_j = scale * q.k_j over visible j, w_j = exp(s_j - max s), o = sum w_j v_j / sum w_j.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = scale * (q @ k.T)
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    return (w @ v) / w.sum(axis=1, keepdims=True)


def attend_additive(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray,
                    scale: float) -> np.ndarray:
    """Softmax attention with an additive mask over every key slot
    ([Horizon] §4: the (c, C) mask is added to the scores, nothing excluded)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = scale * (q @ k.T) + mask
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    return (w @ v) / w.sum(axis=1, keepdims=True)


def causal_attention(q, k, v, scale: float | None = None) -> np.ndarray:
    """One-shot causal prefill ([Glossary] example, the single-pass branch).

    q ``[N, Hq, D]``, k/v ``[N, Hkv, D]`` -> ``[N, Hq, D]`` float64.
    """
    q = np.asarray(q, np.float64)
    n, hq, d = q.shape
    hkv = k.shape[1]
    scale = default_scale(d) if scale is None else scale
    pos = np.arange(n)
    vis = causal_visible(pos, pos)
    out = np.empty((n, hq, d))
    for h in range(hq):
        g = kv_head(h, hq, hkv)
        out[:, h] = attend(q[:, h], k[:, g], v[:, g], vis, scale)
    return out


def chunk_attention(q_chunk, k_seq, v_seq, past_len: int, scale: float | None = None):
    """Attention of one chunk of query rows over the cache ([Wiki] §一.2).

    q_chunk ``[R, Hq, D]`` holds the rows at absolute positions
    past_len .. past_len+R-1.  k_seq/v_seq ``[n, Hkv, D]`` hold the cache in
    position order (slot a = absolute position a) with n >= past_len + R.
    Row i sees keys [0, past_len + i]: the cached prefix [0, past_len) plus its
    own causal triangle.  Returns ``[R, Hq, D]`` float64.
    """
    q_chunk = np.asarray(q_chunk, np.float64)
    r, hq, d = q_chunk.shape
    hkv = k_seq.shape[1]
    n = past_len + r
    scale = default_scale(d) if scale is None else scale
    vis = causal_visible(past_len + np.arange(r), np.arange(n))
    out = np.empty((r, hq, d))
    for h in range(hq):
        g = kv_head(h, hq, hkv)
        out[:, h] = attend(q_chunk[:, h], k_seq[:n, g], v_seq[:n, g], vis, scale)
    return out


# ---------------------------------------------------------------------------
# Contiguous cache at fixed physical capacity
# ---------------------------------------------------------------------------

def new_cache(batch: int, hkv: int, capacity: int, dim: int, dtype=np.float32, fill=0.0):
    """A cache ``[B, Hkv, capacity, D]`` bound at physical capacity ([Wiki] §一.3)."""
    return np.full((batch, hkv, capacity, dim), fill, dtype=dtype)


def kv_append(cache: np.ndarray, new: np.ndarray, past_len) -> np.ndarray:
    """Append rows into a contiguous cache ([Wiki] §一.1).

    cache ``[B, Hkv, cap, D]``; new ``[B, R, Hkv, D]``; row t of sequence b goes
    to slot past_len[b] + t.  Earlier slots are neither read nor rewritten.
    Returns a new array (the input is not modified).
    """
    out = cache.copy()
    b_n, r = new.shape[0], new.shape[1]
    past = np.broadcast_to(np.asarray(past_len), (b_n,))
    for b in range(b_n):
        p = int(past[b])
        if p + r > cache.shape[2]:
            raise ValueError("append past physical capacity")
        out[b, :, p:p + r, :] = np.transpose(new[b], (1, 0, 2))
    return out


def chunked_prefill(q, k, v, W: int, capacity: int | None = None,
                    scale: float | None = None, cache_dtype=None):
    """Chunked prefill of one sequence ([Glossary] example, the chunk loop;
    [Wiki] §一.1 append-only cache).

    q ``[N, Hq, D]``, k/v ``[N, Hkv, D]``.  For each chunk of ``chunk_plan(N, W)``
    the chunk's K/V are appended to a cache of the given physical capacity and
    its rows attend to the cache.  Returns (out ``[N, Hq, D]`` float64,
    list of (k_cache, v_cache) snapshots ``[1, Hkv, cap, D]`` after each chunk,
    chunk sizes).
    """
    n, hq, d = q.shape
    hkv = k.shape[1]
    capacity = n if capacity is None else capacity
    dt = np.asarray(k).dtype if cache_dtype is None else cache_dtype
    kc = new_cache(1, hkv, capacity, d, dt)
    vc = new_cache(1, hkv, capacity, d, dt)
    out = np.empty((n, hq, d))
    snaps = []
    sizes = chunk_plan(n, W)
    start = 0
    for r in sizes:
        kc = kv_append(kc, np.asarray(k[None, start:start + r]), [start])
        vc = kv_append(vc, np.asarray(v[None, start:start + r]), [start])
        k_seq = np.transpose(kc[0], (1, 0, 2))
        v_seq = np.transpose(vc[0], (1, 0, 2))
        out[start:start + r] = chunk_attention(q[start:start + r], k_seq, v_seq, start, scale)
        snaps.append((kc.copy(), vc.copy()))
        start += r
    return out, snaps, sizes


def padded_chunk(q_real, k_real, v_real, kc, vc, past_len: int, W: int,
                 scale: float | None = None):
    """One chunk of a padded prefill ([Wiki] §四).

    The chunk's real rows are widened to ``query_width(r, W)`` by repeating the
    last real row; every widened row is appended and attended; the outputs are
    cut back to the real rows; the valid length is rewound to past_len + r, so
    the pad rows' K/V stay in the slots after it until the next chunk
    overwrites them.  kc/vc ``[1, Hkv, cap, D]``.
    Returns (out ``[r, Hq, D]``, kc, vc, new valid length, rows_padded).
    """
    r = q_real.shape[0]
    rp = query_width(r, W)
    qp = pad_rows(np.asarray(q_real), rp)
    kp = pad_rows(np.asarray(k_real), rp)
    vp = pad_rows(np.asarray(v_real), rp)
    kc = kv_append(kc, kp[None], [past_len])
    vc = kv_append(vc, vp[None], [past_len])
    k_seq = np.transpose(kc[0], (1, 0, 2))
    v_seq = np.transpose(vc[0], (1, 0, 2))
    out = chunk_attention(qp, k_seq, v_seq, past_len, scale)
    return out[:r], kc, vc, past_len + r, rp


# ---------------------------------------------------------------------------
# Right-aligned rolling cache ([Horizon] §2-§5)
# ---------------------------------------------------------------------------

def rolling_update(cache: np.ndarray, new: np.ndarray) -> np.ndarray:
    """[Horizon] §3: concatenate the old cache and the new rows along the
    sequence axis and drop as many of the oldest rows as were added, so the
    cache always holds the newest C positions.  cache ``[H, C, D]``,
    new ``[H, c, D]``."""
    c = new.shape[1]
    return np.concatenate([cache, new], axis=1)[:, c:]


def rolling_mask(c: int, C: int, chunk_idx: int, left_pad: int) -> np.ndarray:
    """Per-chunk additive mask ``[c, C]`` ([Horizon] §4).

    The chunk's c rows are cut from the full causal mask and their key axis is
    right-aligned to the cache length C; everything else is filled with -32768.
    Row i is the query at absolute position p = chunk_idx*c + i.  After the
    chunk is rolled in, cache slot j holds absolute position
    a = (chunk_idx+1)*c - C + j.  The slot is allowed (0) iff it has been
    written (a >= 0), is not a left-pad position (a >= left_pad) and is not in
    the future (a <= p); otherwise it gets -32768.
    """
    p = chunk_idx * c + np.arange(c)
    a = (chunk_idx + 1) * c - C + np.arange(C)
    ok = (a[None, :] >= 0) & (a[None, :] >= left_pad) & (a[None, :] <= p[:, None])
    return np.where(ok, 0.0, MASK_MIN)


def rolling_prefill(q, k, v, c: int, C: int, left_pad: int, scale: float | None = None,
                    cache_dtype=None):
    """Chunk prefill with a right-aligned rolling cache ([Horizon] §3-§5).

    q/k/v ``[L, H, D]`` hold the left-padded sequence (L a multiple of c, the
    first ``left_pad`` positions are pad tokens).  The cache ``[H, C, D]`` starts
    all-zero.  For chunk k: roll the chunk's K/V in, build the (c, C) mask, and
    attend with the mask added to the scores over all C slots.
    Returns (out ``[L, H, D]`` float64, list of (k_cache, v_cache) after each chunk).
    """
    q = np.asarray(q)
    L, h, d = q.shape
    if L % c:
        raise ValueError("aligned length must be a multiple of c")
    if c > C:
        raise ValueError("chunk wider than the cache")
    scale = default_scale(d) if scale is None else scale
    dt = np.asarray(k).dtype if cache_dtype is None else cache_dtype
    kc = np.zeros((h, C, d), dt)
    vc = np.zeros((h, C, d), dt)
    out = np.empty((L, h, d))
    snaps = []
    for ci in range(L // c):
        sl = slice(ci * c, (ci + 1) * c)
        kc = rolling_update(kc, np.transpose(np.asarray(k[sl]), (1, 0, 2)))
        vc = rolling_update(vc, np.transpose(np.asarray(v[sl]), (1, 0, 2)))
        mask = rolling_mask(c, C, ci, left_pad)
        for hh in range(h):
            out[sl, hh] = attend_additive(q[sl, hh], kc[hh], vc[hh], mask, scale)
        snaps.append((kc.copy(), vc.copy()))
    return out, snaps


# ---------------------------------------------------------------------------
# Paged cache ([Glossary] "Related techniques": PagedAttention)
# ---------------------------------------------------------------------------

def paged_write(pool: np.ndarray, table_row, pos: int, kv_row: np.ndarray) -> None:
    """Write one token's K or V ``[Hkv, D]`` at absolute position ``pos`` of a
    sequence whose pages are listed in ``table_row``.  pool
    ``[num_pages, Hkv, page, D]``; the token lands in page
    table_row[pos // page] at offset pos % page.  Modifies ``pool`` in place."""
    page = pool.shape[2]
    pool[int(table_row[pos // page]), :, pos % page, :] = kv_row


def paged_gather(pool: np.ndarray, table_row, n: int) -> np.ndarray:
    """The first ``n`` positions of a paged sequence in position order,
    ``[n, Hkv, D]``."""
    page = pool.shape[2]
    return np.stack([pool[int(table_row[a // page]), :, a % page, :] for a in range(n)])


def mixed_step(q, k_new, v_new, k_pool, v_pool, block_table, rows, past_len,
               scale: float | None = None):
    """One token-budget step over a paged cache ([Glossary] "How chunked prefill works").

    The step's rows are ordered by sequence: sequence s owns ``rows[s]``
    consecutive rows of q ``[T, Hq, D]`` and k_new/v_new ``[T, Hkv, D]`` (one row
    for a decode, a prompt chunk otherwise).  Every row's K/V is appended at
    positions past_len[s] .. past_len[s]+rows[s]-1 first, then each row attends
    causally over its own sequence's cache.  Returns
    (out ``[T, Hq, D]`` float64, k_pool, v_pool, new past lengths).
    """
    kp = k_pool.copy()
    vp = v_pool.copy()
    t = 0
    for s, r in enumerate(rows):
        for i in range(r):
            paged_write(kp, block_table[s], past_len[s] + i, k_new[t + i])
            paged_write(vp, block_table[s], past_len[s] + i, v_new[t + i])
        t += r
    out = np.empty(q.shape, np.float64)
    t = 0
    for s, r in enumerate(rows):
        n = past_len[s] + r
        ks = paged_gather(kp, block_table[s], n)
        vs = paged_gather(vp, block_table[s], n)
        out[t:t + r] = chunk_attention(q[t:t + r], ks, vs, past_len[s], scale)
        t += r
    return out, kp, vp, [p + r for p, r in zip(past_len, rows)]


def attention_row(q_row, k_seq, v_seq, pos: int, scale: float | None = None):
    """Output of a single query row ``[Hq, D]`` at absolute position ``pos`` over a
    cache in position order ``[n, Hkv, D]`` (keys 0..pos).  Used to check sampled
    rows of large workloads one by one."""
    return chunk_attention(np.asarray(q_row)[None], k_seq, v_seq, pos, scale)[0]

