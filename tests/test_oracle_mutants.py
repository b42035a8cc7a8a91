"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin fails for each: a dropped or shifted causal diagonal, a wrong GQA
head map, a wrong scale, a transposed softmax axis, an off-by-one append, a
rolling cache that drops the newest rows, a wrong mask sign or pad bound, a
floor-rounded ladder step, a remainder chunk put first, scores taken against
V, the additive mask left out, a token budget that does not charge the decode
rows, and swapped page indices."""
import math

import numpy as np
import pytest

import oracle.cp_oracle as O
from oracle_pins import ALL_PINS


def _attend_wrong_axis(q, k, v, visible, scale):
    s = scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=0, keepdims=True)
    w = np.nan_to_num(np.exp(s - m))
    return (w @ v) / np.maximum(w.sum(axis=1, keepdims=True), 1e-300)


def _kv_append_off_by_one(cache, new, past_len):
    past = np.asarray(past_len) + 1
    out = cache.copy()
    for b in range(new.shape[0]):
        p = int(np.broadcast_to(past, (new.shape[0],))[b])
        r = min(new.shape[1], cache.shape[2] - p)
        out[b, :, p:p + r, :] = np.transpose(new[b, :r], (1, 0, 2))
    return out


def _rolling_mask_future(c, C, chunk_idx, left_pad):
    p = chunk_idx * c + np.arange(c)
    a = (chunk_idx + 1) * c - C + np.arange(C)
    ok = (a[None, :] >= 0) & (a[None, :] >= left_pad) & (a[None, :] <= p[:, None] + 1)
    return np.where(ok, 0.0, O.MASK_MIN)


def _rolling_mask_pad_inclusive(c, C, chunk_idx, left_pad):
    p = chunk_idx * c + np.arange(c)
    a = (chunk_idx + 1) * c - C + np.arange(C)
    ok = (a[None, :] >= 0) & (a[None, :] >= left_pad - 1) & (a[None, :] <= p[:, None])
    return np.where(ok, 0.0, O.MASK_MIN)


def _ladder_floor(W):
    step = max(1, W // 3)
    out = []
    for i in (1, 2, 3):
        t = i * step
        if t not in out:
            out.append(t)
    return out


def _chunk_plan_remainder_first(n, W):
    s = []
    if n % W:
        s.append(n % W)
    s += [W] * (n // W)
    return s


def _paged_write_swapped(pool, table_row, pos, kv_row):
    page = pool.shape[2]
    pool[int(table_row[pos % page]), :, pos // page % page, :] = kv_row


def _paged_gather_swapped(pool, table_row, n):
    page = pool.shape[2]
    return np.stack([pool[int(table_row[a % page]), :, a // page % page, :] for a in range(n)])


def _attend_scores_from_v(q, k, v, visible, scale):
    s = scale * (np.asarray(q, np.float64) @ np.asarray(v, np.float64).T)
    s = np.where(visible, s, -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w @ np.asarray(v, np.float64)) / w.sum(axis=1, keepdims=True)


def _attend_additive_mask_dropped(q, k, v, mask, scale):
    s = scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w @ np.asarray(v, np.float64)) / w.sum(axis=1, keepdims=True)


def _schedule_budget_ignores_decodes(budget, n_running, prompt_lens):
    decodes = list(range(n_running))
    done = [0] * len(prompt_lens)
    steps = []
    while any(d < n for d, n in zip(done, prompt_lens)):
        left = budget  # the mistake: decode rows not charged
        chunks, finished = [], []
        for i, n in enumerate(prompt_lens):
            if done[i] >= n or left == 0:
                continue
            take = min(left, n - done[i])
            chunks.append((n_running + i, done[i], take))
            done[i] += take
            left -= take
            if done[i] == n:
                finished.append(n_running + i)
        steps.append((list(decodes), chunks))
        decodes += finished
    return steps


MUTANTS = {
    "diag_dropped": ("causal_visible", lambda pq, pk: pk[None, :] < pq[:, None]),
    "future_leak": ("causal_visible", lambda pq, pk: pk[None, :] <= pq[:, None] + 1),
    "gqa_modulo": ("kv_head", lambda h, hq, hkv: h % hkv),
    "scale_1_over_d": ("default_scale", lambda d: 1.0 / d),
    "scale_missing": ("default_scale", lambda d: 1.0),
    "softmax_axis": ("attend", _attend_wrong_axis),
    "append_off_by_one": ("kv_append", _kv_append_off_by_one),
    "rolling_drops_newest": ("rolling_update",
                             lambda cache, new: np.concatenate([cache, new], axis=1)[:, :cache.shape[1]]),
    "rolling_mask_future": ("rolling_mask", _rolling_mask_future),
    "rolling_mask_pad": ("rolling_mask", _rolling_mask_pad_inclusive),
    "ladder_floor": ("query_ladder", _ladder_floor),
    "remainder_first": ("chunk_plan", _chunk_plan_remainder_first),
    "scores_from_v": ("attend", _attend_scores_from_v),
    "additive_mask_dropped": ("attend_additive", _attend_additive_mask_dropped),
    "budget_ignores_decodes": ("schedule", _schedule_budget_ignores_decodes),
    "pad_with_zeros": ("pad_rows", lambda x, rp: np.concatenate(
        [x, np.zeros((rp - x.shape[0],) + x.shape[1:], x.dtype)])),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception as e:  # AssertionError or a shape error both count
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"no pin caught mutant {name}"


def test_paged_swap_is_caught(monkeypatch):
    monkeypatch.setattr(O, "paged_write", _paged_write_swapped)
    monkeypatch.setattr(O, "paged_gather", _paged_gather_swapped)
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception as e:
            failed.append(pin.__name__)
    assert failed
