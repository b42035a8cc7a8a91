"""Helpers for the GPU parity tests: drive the C ABI through the binding and
convert tensors for the oracle.  No attention arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

import chunked_prefill_causal_cp_gb300 as cp

BF16_TOL = 2e-2   # max-abs bound for 16-bit inputs with fp32 accumulation
F32_TOL = 1e-4    # max-abs bound for the fp32 path


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


class Contig:
    """A contiguous cache at fixed physical capacity plus its valid length."""

    def __init__(self, dtype, hq, hkv, d, cap, batch=1, poison=True, dev="cuda", fused=False):
        self.desc = cp.layer_desc(dtype, batch, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=cap)
        fill = float("nan") if poison else 0.0
        self.k = torch.full((batch, hkv, cap, d), fill, dtype=dtype, device=dev)
        self.v = torch.full((batch, hkv, cap, d), fill, dtype=dtype, device=dev)
        self.lens = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.cap = cap
        self.fused = fused  # one cp_prefill_chunk call per chunk instead of append + attention
        # room for the split-KV partials of up to 16 rows per sequence (short chunks take that path)
        self.ws = torch.zeros(max(cp.cp_workspace_size(self.desc, batch * 16, cap, batch), 16), dtype=torch.uint8,
                              device=dev)

    def chunk(self, q, k_new, v_new, real_rows, past, out=None):
        """Append a [B, R, ...] chunk, attend, commit real_rows.  Returns out [B, R, Hq, D]."""
        R = q.shape[1]
        if out is None:
            out = torch.empty_like(q)
        if self.fused:
            cp.cp_prefill_chunk(self.desc, q, k_new, v_new, self.k, self.v, self.lens, R, real_rows, past, out,
                                self.ws, dev_status=self.status)
            return out
        cp.cp_kv_append(self.desc, k_new, v_new, R, self.k, self.v, self.lens, past,
                        dev_status=self.status)
        cp.cp_prefill_chunk_attn(self.desc, q, self.k, self.v, self.lens, R, real_rows, past, out,
                                 self.ws, commit=True, dev_status=self.status)
        return out


def prefill(cache: Contig, q, k, v, W, pad=False):
    """Chunked prefill of one prompt [N, H, D] (batch 1).  Returns (out [N,Hq,D],
    list of rows_padded used).  With pad=True each chunk is widened to its
    ladder tier by repeating the last real row."""
    n = q.shape[0]
    out = torch.empty_like(q)
    widths = []
    past = 0
    for r in cp.cp_chunk_plan(n, W):
        sl = slice(past, past + r)
        if pad:
            rp = cp.cp_query_width(r, W)
            idx = torch.cat([torch.arange(past, past + r), torch.full((rp - r,), past + r - 1)]).to(q.device)
            qc, kc, vc = q[idx], k[idx], v[idx]
        else:
            rp = r
            qc, kc, vc = q[sl], k[sl], v[sl]
        o = cache.chunk(qc[None].contiguous(), kc[None].contiguous(), vc[None].contiguous(), r, past)
        out[sl] = o[0, :r]
        widths.append(rp)
        past += r
    return out, widths
