"""The C++ oracle against the numpy oracle on the same random inputs (both
are pinned on their own in test_oracle.py), and the C++ oracle's thread count
does not change a single bit of its results (each (row, head) pair is
computed start to finish by one thread)."""
import numpy as np
import pytest

import oracle.cp_oracle as N
import oracle.cpp as C


@pytest.fixture(autouse=True)
def _threads():
    C.set_threads(0)
    yield
    C.set_threads(0)


def _rng(seed):
    return np.random.default_rng(seed)


def test_chunked_prefill_matches_numpy():
    rng = _rng(31)
    q = rng.standard_normal((45, 8, 16))
    k = rng.standard_normal((45, 2, 16))
    v = rng.standard_normal((45, 2, 16))
    for W in (1, 7, 45, 64):
        a, sa, za = N.chunked_prefill(q, k, v, W, capacity=50)
        b, sb, zb = C.chunked_prefill(q, k, v, W, capacity=50)
        assert za == zb
        assert np.allclose(a, b, rtol=0, atol=1e-12)
        for (ka, va), (kb, vb) in zip(sa, sb):
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def test_rolling_prefill_matches_numpy():
    rng = _rng(32)
    L, c, cap, lp = 48, 8, 20, 5
    q = rng.standard_normal((L, 3, 8))
    k = rng.standard_normal((L, 3, 8))
    v = rng.standard_normal((L, 3, 8))
    a, sa = N.rolling_prefill(q, k, v, c, cap, lp)
    b, sb = C.rolling_prefill(q, k, v, c, cap, lp)
    assert np.allclose(a, b, rtol=0, atol=1e-12)
    for (ka, va), (kb, vb) in zip(sa, sb):
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    for ci in range(L // c):
        assert np.array_equal(N.rolling_mask(c, cap, ci, lp), C.rolling_mask(c, cap, ci, lp))


def test_mixed_step_and_padding_match_numpy():
    rng = _rng(33)
    page, hq, hkv, d = 4, 4, 2, 8
    rows, past = [1, 1, 6], [5, 9, 3]
    table = rng.permutation(24).astype(np.int32).reshape(3, 8)
    kp = rng.standard_normal((24, hkv, page, d))
    vp = rng.standard_normal((24, hkv, page, d))
    T = sum(rows)
    q = rng.standard_normal((T, hq, d))
    kn = rng.standard_normal((T, hkv, d))
    vn = rng.standard_normal((T, hkv, d))
    oa, ka, va, pa = N.mixed_step(q, kn, vn, kp, vp, table, rows, past)
    ob, kb, vb, pb = C.mixed_step(q, kn, vn, kp, vp, table, rows, past)
    assert pa == pb and np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert np.allclose(oa, ob, rtol=0, atol=1e-12)
    kc = np.zeros((1, hkv, 40, d))
    r = 5
    ra = N.padded_chunk(q[:r], kn[:r], vn[:r], kc, kc.copy(), 3, 12)
    rb = C.padded_chunk(q[:r], kn[:r], vn[:r], kc, kc.copy(), 3, 12)
    assert np.allclose(ra[0], rb[0], rtol=0, atol=1e-12)
    assert np.array_equal(ra[1], rb[1]) and ra[3:] == rb[3:]
    x = rng.standard_normal((5, 3, 2)).astype(np.float32)
    assert np.array_equal(N.pad_rows(x, 9), C.pad_rows(x, 9))


def test_schedules_match_numpy():
    for budget, nrun, prompts in [(8192, 64, [20000] * 4), (2048, 64, [20000] * 4), (37, 5, [100, 3, 50, 1]),
                                  (300, 0, [1000, 999]), (10, 3, [9, 4])]:
        assert N.schedule(budget, nrun, prompts) == C.schedule(budget, nrun, prompts)


def test_thread_count_changes_no_bit():
    rng = _rng(34)
    q = rng.standard_normal((60, 8, 16))
    k = rng.standard_normal((60, 2, 16))
    v = rng.standard_normal((60, 2, 16))
    C.set_threads(1)
    one, _, _ = C.chunked_prefill(q, k, v, 16)
    C.set_threads(5)
    five, _, _ = C.chunked_prefill(q, k, v, 16)
    assert np.array_equal(one, five)
