"""Python binding of libcp.so, the GB300 chunked-prefill causal attention library.

Argument marshalling only: each function takes torch tensors (device memory
allocated by the caller), passes their pointers to the C entry point of the
same name declared in ``include/cp_api.h``, and raises ``CPError`` on a
non-zero status.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback of any kind.  If the library has not been
built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_size_t, c_void_p

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcp.so")

CP_OK = 0
CP_ERR_INVALID_ARG = -1
CP_ERR_UNSUPPORTED = -2
CP_ERR_CAPACITY = -3
CP_ERR_CUDA = -4
CP_ERR_WORKSPACE = -5
CP_DEV_BOUNDS = 1
CP_DEV_TIMEOUT = 2

CP_F32, CP_BF16, CP_F16 = 0, 1, 2
CP_CACHE_CONTIG, CP_CACHE_ROLLING, CP_CACHE_PAGED = 0, 1, 2

DTYPE_CODE = {torch.float32: CP_F32, torch.bfloat16: CP_BF16, torch.float16: CP_F16}


class LayerDesc(ctypes.Structure):
    """Mirror of ``cp_layer_desc``."""

    _fields_ = [
        ("dtype", c_int32), ("batch", c_int32), ("num_q_heads", c_int32),
        ("num_kv_heads", c_int32), ("head_dim", c_int32), ("kind", c_int32),
        ("capacity", c_int32), ("page_size", c_int32), ("num_pages", c_int32),
        ("max_blocks", c_int32), ("scale", c_float),
    ]


class SchedEntry(ctypes.Structure):
    """Mirror of ``cp_sched_entry``."""

    _fields_ = [("step", c_int32), ("seq", c_int32), ("start", c_int32), ("rows", c_int32)]


class CPError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {cp_status_string(status)} ({status})")
        self.status = status


_lib = None


def lib():
    """The loaded libcp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = c_void_p
        L.cp_kv_append.argtypes = [POINTER(LayerDesc), P, P, c_int32, P, P, P, P, c_int32, P, P]
        L.cp_pad_chunk.argtypes = [POINTER(LayerDesc), P, P, P, c_int32, c_int32, P]
        L.cp_prefill_chunk_attn.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, c_int32, c_int32,
                                            c_int32, P, P, c_size_t, c_int32, P, P]
        L.cp_prefill_chunk.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, P, c_int32, c_int32,
                                       c_int32, P, P, c_size_t, P, P]
        L.cp_mixed_step.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, P, c_int32, c_int32,
                                    c_int32, P, P, c_size_t, P, P]
        L.cp_mixed_step_overlap.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, P, c_int32, c_int32,
                                            c_int32, P, P, c_size_t, P, P, P, P, P]
        L.cp_prefill_varlen.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, c_int32, c_int32, c_int32, P,
                                        P, c_size_t, P, P]
        L.cp_prefill_varlen_overlap.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, c_int32, c_int32,
                                                c_int32, P, P, c_size_t, P, P, P, P, P]
        L.cp_mixed_step_noalloc.argtypes = [POINTER(LayerDesc), P, P, P, P, P, P, P, P, c_int32, c_int32,
                                            c_int32, P, P, P]
        L.cp_mixed_step_noalloc.restype = c_int32
        L.cp_noalloc_scratch_bytes.argtypes = []
        L.cp_noalloc_scratch_bytes.restype = c_size_t
        L.cp_workspace_size.argtypes = [POINTER(LayerDesc), c_int32, c_int32, c_int32]
        L.cp_workspace_size.restype = c_size_t
        L.cp_chunk_plan.argtypes = [c_int32, c_int32, POINTER(c_int32), c_int32]
        L.cp_query_ladder.argtypes = [c_int32, POINTER(c_int32)]
        L.cp_query_width.argtypes = [c_int32, c_int32]
        L.cp_aligned_length.argtypes = [c_int32, c_int32]
        L.cp_rolling_mask.argtypes = [c_int32, c_int32, c_int32, c_int32, POINTER(c_float)]
        L.cp_schedule.argtypes = [c_int32, c_int32, POINTER(c_int32), c_int32, POINTER(SchedEntry), c_int32]
        L.cp_status_string.argtypes = [c_int32]
        L.cp_selftest_bounded_wait.argtypes = [P, P, P]
        L.cp_abi_version.argtypes = []
        L.cp_status_string.restype = ctypes.c_char_p
        for name in ("cp_kv_append", "cp_pad_chunk", "cp_prefill_chunk_attn", "cp_prefill_chunk",
                     "cp_mixed_step", "cp_mixed_step_overlap", "cp_prefill_varlen", "cp_prefill_varlen_overlap",
                     "cp_chunk_plan",
                     "cp_query_ladder", "cp_query_width", "cp_aligned_length", "cp_rolling_mask",
                     "cp_schedule", "cp_abi_version", "cp_selftest_bounded_wait"):
            getattr(L, name).restype = c_int32
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    for t in tensors:
        if isinstance(t, torch.Tensor) and t.is_cuda:
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _check(status: int, where: str):
    if status != CP_OK:
        raise CPError(status, where)


def layer_desc(dtype, batch, num_q_heads, num_kv_heads, head_dim, kind=CP_CACHE_CONTIG,
               capacity=0, page_size=0, num_pages=0, max_blocks=0, scale=0.0) -> LayerDesc:
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return LayerDesc(code, batch, num_q_heads, num_kv_heads, head_dim, kind, capacity, page_size,
                     num_pages, max_blocks, scale)


def cp_kv_append(desc, k_new, v_new, rows, k_cache, v_cache, seqlens_k, max_past,
                 block_table=None, dev_status=None, stream=None):
    s = lib().cp_kv_append(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), rows, _ptr(k_cache),
                           _ptr(v_cache), _ptr(seqlens_k), _ptr(block_table), max_past,
                           _ptr(dev_status), _stream(stream, k_new))
    _check(s, "cp_kv_append")


def cp_pad_chunk(desc, q, k_new, v_new, real_rows, rows_padded, stream=None):
    s = lib().cp_pad_chunk(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), real_rows, rows_padded,
                           _stream(stream, q, k_new, v_new))
    _check(s, "cp_pad_chunk")


def cp_prefill_chunk_attn(desc, q, k_cache, v_cache, seqlens_k, rows_padded, real_rows, max_past,
                          out, workspace=None, commit=True, block_table=None, left_pad=None,
                          dev_status=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = lib().cp_prefill_chunk_attn(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(seqlens_k), _ptr(block_table), _ptr(left_pad), rows_padded,
                                    real_rows, max_past, _ptr(out), _ptr(workspace), ws_bytes,
                                    1 if commit else 0, _ptr(dev_status), _stream(stream, q))
    _check(s, "cp_prefill_chunk_attn")


def cp_prefill_chunk(desc, q, k_new, v_new, k_cache, v_cache, seqlens_k, rows_padded, real_rows, max_past,
                     out, workspace, block_table=None, left_pad=None, dev_status=None, stream=None):
    """Append, attention and commit of one chunk in one call (see include/cp_api.h)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = lib().cp_prefill_chunk(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                               _ptr(v_cache), _ptr(seqlens_k), _ptr(block_table), _ptr(left_pad), rows_padded,
                               real_rows, max_past, _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status),
                               _stream(stream, q))
    _check(s, "cp_prefill_chunk")


def cp_mixed_step(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len,
                  num_seqs, total_rows, max_ctx, out, workspace, dev_status=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = lib().cp_mixed_step(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                            _ptr(v_pages), _ptr(block_table), _ptr(cu_rows), _ptr(past_len), num_seqs,
                            total_rows, max_ctx, _ptr(out), _ptr(workspace), ws_bytes,
                            _ptr(dev_status), _stream(stream, q))
    _check(s, "cp_mixed_step")


def _side_handles(side_stream, fork_event, join_event):
    """Raw handles of a side stream and two events (torch objects or raw handles)."""
    side = side_stream if isinstance(side_stream, int) else side_stream.cuda_stream
    evs = []
    for ev in (fork_event, join_event):
        if isinstance(ev, int):
            evs.append(ev)
            continue
        if not ev.cuda_event:  # torch creates the event on its first record
            ev.record(side_stream if not isinstance(side_stream, int) else None)
        evs.append(ev.cuda_event)
    return side, evs


def cp_mixed_step_overlap(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len,
                          num_seqs, total_rows, max_ctx, out, workspace, side_stream, fork_event, join_event,
                          dev_status=None, stream=None):
    """cp_mixed_step with the split-KV kernels on `side_stream` beside the
    tensor-core kernel (see include/cp_api.h).  `side_stream` is a
    torch.cuda.Stream (or a raw handle); the events are torch.cuda.Event
    objects (or raw handles)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    side, evs = _side_handles(side_stream, fork_event, join_event)
    s = lib().cp_mixed_step_overlap(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                    _ptr(v_pages), _ptr(block_table), _ptr(cu_rows), _ptr(past_len), num_seqs,
                                    total_rows, max_ctx, _ptr(out), _ptr(workspace), ws_bytes,
                                    _ptr(dev_status), _stream(stream, q), side, evs[0], evs[1])
    _check(s, "cp_mixed_step_overlap")


def cp_prefill_varlen(desc, q, k_new, v_new, k_cache, v_cache, cu_rows, seqlens_k, num_seqs, total_rows, max_ctx,
                      out, workspace, dev_status=None, stream=None):
    """Several sequences with ragged rows over a contiguous cache in one call (see include/cp_api.h)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = lib().cp_prefill_varlen(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                _ptr(v_cache), _ptr(cu_rows), _ptr(seqlens_k), num_seqs, total_rows, max_ctx,
                                _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream, q))
    _check(s, "cp_prefill_varlen")


def cp_prefill_varlen_overlap(desc, q, k_new, v_new, k_cache, v_cache, cu_rows, seqlens_k, num_seqs, total_rows,
                              max_ctx, out, workspace, side_stream, fork_event, join_event, dev_status=None,
                              stream=None):
    """cp_prefill_varlen with the one-row sequences' split-KV kernels on
    `side_stream` (see include/cp_api.h); handles as in cp_mixed_step_overlap."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    side, evs = _side_handles(side_stream, fork_event, join_event)
    s = lib().cp_prefill_varlen_overlap(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(cu_rows), _ptr(seqlens_k), num_seqs, total_rows,
                                        max_ctx, _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                        _stream(stream, q), side, evs[0], evs[1])
    _check(s, "cp_prefill_varlen_overlap")


def cp_mixed_step_noalloc(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len,
                          num_seqs, total_rows, max_ctx, out, dev_status=None, stream=None):
    """cp_mixed_step without a workspace: the split-KV scratch is a fixed array
    inside the library (see include/cp_api.h for its limit and sharing rules)."""
    s = lib().cp_mixed_step_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                    _ptr(v_pages), _ptr(block_table), _ptr(cu_rows), _ptr(past_len),
                                    num_seqs, total_rows, max_ctx, _ptr(out), _ptr(dev_status),
                                    _stream(stream, q))
    _check(s, "cp_mixed_step_noalloc")


def cp_noalloc_scratch_bytes() -> int:
    return int(lib().cp_noalloc_scratch_bytes())


def cp_workspace_size(desc, max_rows, max_ctx, num_seqs) -> int:
    return int(lib().cp_workspace_size(ctypes.byref(desc), max_rows, max_ctx, num_seqs))


def cp_chunk_plan(n_tokens, chunk):
    n = lib().cp_chunk_plan(n_tokens, chunk, None, 0)
    _check(min(n, 0), "cp_chunk_plan")
    buf = (c_int32 * max(n, 1))()
    lib().cp_chunk_plan(n_tokens, chunk, buf, n)
    return list(buf[:n])


def cp_query_ladder(chunk):
    buf = (c_int32 * 3)()
    n = lib().cp_query_ladder(chunk, buf)
    _check(min(n, 0), "cp_query_ladder")
    return list(buf[:n])


def cp_query_width(real_rows, chunk):
    w = lib().cp_query_width(real_rows, chunk)
    _check(min(w, 0), "cp_query_width")
    return w


def cp_aligned_length(n_real, c):
    v = lib().cp_aligned_length(n_real, c)
    _check(min(v, 0), "cp_aligned_length")
    return v


def cp_rolling_mask(c, C, chunk_idx, left_pad):
    buf = (c_float * (c * C))()
    _check(lib().cp_rolling_mask(c, C, chunk_idx, left_pad, buf), "cp_rolling_mask")
    return torch.frombuffer(bytearray(buf), dtype=torch.float32).reshape(c, C)


def cp_schedule(budget, n_running, prompt_lens):
    arr = (c_int32 * max(len(prompt_lens), 1))(*prompt_lens)
    n = lib().cp_schedule(budget, n_running, arr, len(prompt_lens), None, 0)
    _check(min(n, 0), "cp_schedule")
    buf = (SchedEntry * max(n, 1))()
    lib().cp_schedule(budget, n_running, arr, len(prompt_lens), buf, n)
    return [(e.step, e.seq, e.start, e.rows) for e in buf[:n]]


def cp_status_string(status) -> str:
    return lib().cp_status_string(status).decode()


def cp_abi_version() -> int:
    return lib().cp_abi_version()


def cp_selftest_bounded_wait(dev_status, dev_out, stream=None) -> int:
    return lib().cp_selftest_bounded_wait(_ptr(dev_status), _ptr(dev_out), _stream(stream, dev_out))
