"""The C++ oracle (``cp_oracle.cpp``) behind the same Python interface as the
numpy oracle in ``cp_oracle.py``.

TEST INFRASTRUCTURE ONLY: the same import rules as the rest of ``oracle/``.
This module only marshals numpy arrays to float64 / int32 buffers and back;
every step of the arithmetic runs in the C++ library, which ``build()``
compiles with g++ (no CUDA) on first use.

``set_threads(n)`` fixes the number of std::threads the attention functions
use (0: every hardware thread).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cp_oracle.cpp")
LIB = os.path.join(HERE, "libcp_oracle.so")
MASK_MIN = -32768.0

_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle library next to its source (plain g++, -O2, no
    fast-math, so every sum keeps its written order)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


def load(path: str):
    """The oracle library at `path` with every function's signature set (the
    tests also load variant builds of the same source through this)."""
    L = ctypes.CDLL(path)
    sig = {
        "cpo_set_threads": (None, [ctypes.c_int]),
        "cpo_threads": (ctypes.c_int, []),
        "cpo_chunk_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I, ctypes.c_int]),
        "cpo_query_ladder": (ctypes.c_int, [ctypes.c_int, _I]),
        "cpo_query_width": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
        "cpo_left_pad_length": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
        "cpo_schedule": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I, ctypes.c_int, _I, ctypes.c_int]),
        "cpo_pad_rows": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_int64, ctypes.c_int, _D]),
        "cpo_chunk_attention": (None, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D,
                                       ctypes.c_int, ctypes.c_double, _D]),
        "cpo_causal_attention": (None, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D,
                                        ctypes.c_double, _D]),
        "cpo_chunked_prefill": (ctypes.c_int, [_D, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _D,
                                               _D, _D, _D]),
        "cpo_kv_append": (ctypes.c_int, [_D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _I]),
        "cpo_padded_chunk": (ctypes.c_int, [_D, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, _D]),
        "cpo_rolling_update": (None, [_D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D]),
        "cpo_rolling_mask": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D]),
        "cpo_rolling_prefill": (ctypes.c_int, [_D, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                               _D, _D]),
        "cpo_paged_write": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I,
                                           ctypes.c_int, _D]),
        "cpo_paged_gather": (ctypes.c_int, [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I,
                                            ctypes.c_int, _D]),
        "cpo_mixed_step": (ctypes.c_int, [_D, _D, _D, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, _I, ctypes.c_int, _I, _I, ctypes.c_int,
                                          ctypes.c_double, _D]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def set_threads(n: int) -> None:
    lib().cpo_set_threads(int(n))


def threads() -> int:
    return int(lib().cpo_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dp(a):
    return a.ctypes.data_as(_D)


def _ip(a):
    return a.ctypes.data_as(_I)


def _scale(scale):
    return 0.0 if scale is None else float(scale)


# ---------------------------------------------------------------- plans

def chunk_plan(n_tokens: int, W: int) -> list[int]:
    n = lib().cpo_chunk_plan(int(n_tokens), int(W), None, 0)
    if n < 0:
        raise ValueError("W must be positive and n_tokens non-negative")
    buf = np.zeros(max(n, 1), np.int32)
    lib().cpo_chunk_plan(int(n_tokens), int(W), _ip(buf), n)
    return [int(x) for x in buf[:n]]


def query_ladder(W: int) -> list[int]:
    buf = np.zeros(3, np.int32)
    n = lib().cpo_query_ladder(int(W), _ip(buf))
    if n < 0:
        raise ValueError("W must be positive")
    return [int(x) for x in buf[:n]]


def query_width(real_rows: int, W: int) -> int:
    w = lib().cpo_query_width(int(real_rows), int(W))
    if w < 0:
        raise ValueError("real_rows must be in [1, W]")
    return int(w)


def left_pad_length(n_real: int, c: int) -> int:
    return int(lib().cpo_left_pad_length(int(n_real), int(c)))


def schedule(budget: int, n_running: int, prompt_lens: list[int]):
    """Same return form as the numpy oracle: ``[(decode_ids, [(seq, start, rows), ...]), ...]``."""
    pl = _i32(list(prompt_lens) or [0])
    n = lib().cpo_schedule(int(budget), int(n_running), _ip(pl), len(prompt_lens), None, 0)
    if n < 0:
        raise ValueError("budget leaves no room for prompt tokens" if n == -2 else "invalid arguments")
    buf = np.zeros((max(n, 1), 4), np.int32)
    lib().cpo_schedule(int(budget), int(n_running), _ip(pl), len(prompt_lens), _ip(buf), n)
    steps: dict[int, tuple[list, list]] = {}
    for st, seq, start, rows in buf[:n].tolist():
        d, chunks = steps.setdefault(st, ([], []))
        if start < 0:
            d.append(seq)
        else:
            chunks.append((seq, start, rows))
    return [steps[i] for i in sorted(steps)]


def pad_rows(x: np.ndarray, rows_padded: int) -> np.ndarray:
    x = np.asarray(x)
    r = x.shape[0]
    if rows_padded < r:
        raise ValueError("rows_padded < rows")
    xf = _f64(x).reshape(r, -1)
    out = np.empty((rows_padded, xf.shape[1]), np.float64)
    if lib().cpo_pad_rows(_dp(xf), r, xf.shape[1], int(rows_padded), _dp(out)) != 0:
        raise ValueError("bad arguments")
    return out.reshape((rows_padded,) + x.shape[1:]).astype(x.dtype)


# ---------------------------------------------------------------- attention

def chunk_attention(q_chunk, k_seq, v_seq, past_len: int, scale: float | None = None):
    q = _f64(q_chunk)
    r, hq, d = q.shape
    n = int(past_len) + r
    k = _f64(np.asarray(k_seq)[:n])
    v = _f64(np.asarray(v_seq)[:n])
    out = np.empty((r, hq, d), np.float64)
    lib().cpo_chunk_attention(_dp(q), r, hq, k.shape[1], d, _dp(k), _dp(v), int(past_len), _scale(scale), _dp(out))
    return out


def causal_attention(q, k, v, scale: float | None = None) -> np.ndarray:
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, hq, d = q.shape
    out = np.empty((n, hq, d), np.float64)
    lib().cpo_causal_attention(_dp(q), n, hq, k.shape[1], d, _dp(k), _dp(v), _scale(scale), _dp(out))
    return out


def attention_row(q_row, k_seq, v_seq, pos: int, scale: float | None = None):
    return chunk_attention(np.asarray(q_row)[None], k_seq, v_seq, pos, scale)[0]


# ---------------------------------------------------------------- contiguous cache

def new_cache(batch: int, hkv: int, capacity: int, dim: int, dtype=np.float32, fill=0.0):
    return np.full((batch, hkv, capacity, dim), fill, dtype=dtype)


def kv_append(cache: np.ndarray, new: np.ndarray, past_len) -> np.ndarray:
    cache = np.asarray(cache)
    c = _f64(cache).copy()
    nw = _f64(new)
    b, r = nw.shape[0], nw.shape[1]
    past = _i32(np.broadcast_to(np.asarray(past_len), (b,)))
    if lib().cpo_kv_append(_dp(c), _dp(nw), b, r, c.shape[1], c.shape[2], c.shape[3], _ip(past)) != 0:
        raise ValueError("append past physical capacity")
    return c.astype(cache.dtype)


def chunked_prefill(q, k, v, W: int, capacity: int | None = None, scale: float | None = None, cache_dtype=None):
    dt = np.asarray(k).dtype if cache_dtype is None else cache_dtype
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, hq, d = q.shape
    hkv = k.shape[1]
    cap = n if capacity is None else int(capacity)
    sizes = chunk_plan(n, W)
    out = np.empty((n, hq, d), np.float64)
    kc = np.empty((hkv, cap, d), np.float64)
    vc = np.empty((hkv, cap, d), np.float64)
    snaps = np.empty((max(len(sizes), 1), 2, hkv, cap, d), np.float64)
    rc = lib().cpo_chunked_prefill(_dp(q), _dp(k), _dp(v), n, hq, hkv, d, int(W), cap, _scale(scale), _dp(out),
                                   _dp(kc), _dp(vc), _dp(snaps))
    if rc < 0:
        raise ValueError("invalid arguments")
    snap_list = [(snaps[i, 0][None].astype(dt), snaps[i, 1][None].astype(dt)) for i in range(len(sizes))]
    return out, snap_list, sizes


def padded_chunk(q_real, k_real, v_real, kc, vc, past_len: int, W: int, scale: float | None = None):
    dt = np.asarray(kc).dtype
    q, k, v = _f64(q_real), _f64(k_real), _f64(v_real)
    r, hq, d = q.shape
    hkv = k.shape[1]
    kcf = _f64(kc)[0].copy()
    vcf = _f64(vc)[0].copy()
    cap = kcf.shape[1]
    rp = query_width(r, W)
    out = np.empty((rp, hq, d), np.float64)
    got = lib().cpo_padded_chunk(_dp(q), _dp(k), _dp(v), r, hq, hkv, d, _dp(kcf), _dp(vcf), cap, int(past_len),
                                 int(W), _scale(scale), _dp(out))
    if got != rp:
        raise ValueError("invalid arguments")
    return out[:r], kcf[None].astype(dt), vcf[None].astype(dt), int(past_len) + r, rp


# ---------------------------------------------------------------- rolling cache

def rolling_update(cache: np.ndarray, new: np.ndarray) -> np.ndarray:
    dt = np.asarray(cache).dtype
    c0, n0 = _f64(cache), _f64(new)
    h, C, d = c0.shape
    out = np.empty_like(c0)
    lib().cpo_rolling_update(_dp(c0), _dp(n0), h, C, n0.shape[1], d, _dp(out))
    return out.astype(dt)


def rolling_mask(c: int, C: int, chunk_idx: int, left_pad: int) -> np.ndarray:
    out = np.empty((c, C), np.float64)
    lib().cpo_rolling_mask(int(c), int(C), int(chunk_idx), int(left_pad), _dp(out))
    return out


def rolling_prefill(q, k, v, c: int, C: int, left_pad: int, scale: float | None = None, cache_dtype=None):
    dt = np.asarray(k).dtype if cache_dtype is None else cache_dtype
    q, k, v = _f64(q), _f64(k), _f64(v)
    L, h, d = q.shape
    if c <= 0 or L % c:
        raise ValueError("aligned length must be a multiple of c")
    if c > C:
        raise ValueError("chunk wider than the cache")
    out = np.empty((L, h, d), np.float64)
    snaps = np.empty((max(L // c, 1), 2, h, C, d), np.float64)
    if lib().cpo_rolling_prefill(_dp(q), _dp(k), _dp(v), L, h, d, int(c), int(C), int(left_pad), _scale(scale),
                                 _dp(out), _dp(snaps)) < 0:
        raise ValueError("invalid arguments")
    return out, [(snaps[i, 0].astype(dt), snaps[i, 1].astype(dt)) for i in range(L // c)]


# ---------------------------------------------------------------- paged cache

def paged_write(pool: np.ndarray, table_row, pos: int, kv_row: np.ndarray) -> None:
    """In place, like the numpy oracle (the pool must be a float64 array)."""
    if pool.dtype != np.float64 or not pool.flags["C_CONTIGUOUS"]:
        raise TypeError("the C++ oracle writes float64 C-contiguous pools in place")
    tr = _i32(table_row)
    row = _f64(kv_row)
    P, hkv, page, d = pool.shape
    if lib().cpo_paged_write(_dp(pool), P, hkv, page, d, _ip(tr), int(pos), _dp(row)) != 0:
        raise IndexError("page id out of range")


def paged_gather(pool: np.ndarray, table_row, n: int) -> np.ndarray:
    p = _f64(pool)
    tr = _i32(table_row)
    P, hkv, page, d = p.shape
    out = np.empty((int(n), hkv, d), np.float64)
    if lib().cpo_paged_gather(_dp(p), P, hkv, page, d, _ip(tr), int(n), _dp(out)) != 0:
        raise IndexError("page id out of range")
    return out


def mixed_step(q, k_new, v_new, k_pool, v_pool, block_table, rows, past_len, scale: float | None = None):
    q, kn, vn = _f64(q), _f64(k_new), _f64(v_new)
    kp = _f64(k_pool).copy()
    vp = _f64(v_pool).copy()
    bt = _i32(block_table)
    rw = _i32(rows)
    past = _i32(past_len).copy()
    P, hkv, page, d = kp.shape
    out = np.empty(q.shape, np.float64)
    if lib().cpo_mixed_step(_dp(q), _dp(kn), _dp(vn), _dp(kp), _dp(vp), P, q.shape[1], hkv, page, d, _ip(bt),
                            bt.shape[1], _ip(rw), _ip(past), len(rows), _scale(scale), _dp(out)) != 0:
        raise IndexError("page id out of range")
    return out, kp, vp, [int(x) for x in past]
