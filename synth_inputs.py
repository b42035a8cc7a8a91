"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and builds integer layouts (prompt
lengths, page permutations).  It holds none of the attention arithmetic, so
the CPU oracle and the CUDA path can both be fed from it without sharing any
of the method's code.

All tensors are drawn on the CPU with an explicit ``torch.Generator`` so the
same seed gives the same values on every machine.

Workloads (sizes follow the five configurations of the chunked-prefill
problem; every seed is fixed here):

  * ``fp32_sdpa_example``  1 x 8 heads x 64 dims, 1000 tokens, fp32, drawn the
    way the Ultralytics glossary page "Chunked Prefill" draws its one-layer
    example (seed 0, one (3, 1, 8, 1000, 64) normal tensor split into q, k, v).
  * ``gqa_prompt``         GQA 32/8 heads, head_dim 128, bf16 N(0,1) prompt.
  * ``ladder_prompts``     the prompt lengths {1041,1468,3118,3788,1137,1200}.
  * ``rolling_prompt``     16 heads, head_dim 128, fp16, left-padded prompt.
  * ``mixed_batch``        64 decode contexts U{512..8192} in 16-token pages
                           plus 4 prompts of 20000 tokens.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

__all__ = [
    "normal",
    "fp32_sdpa_example",
    "gqa_prompt",
    "LADDER_PROMPT_LENGTHS",
    "ladder_prompt",
    "rolling_prompt",
    "MixedBatch",
    "mixed_batch",
]

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def normal(shape, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """iid N(0,1) values of ``shape`` drawn on the CPU from ``seed``, cast to ``dtype``."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def fp32_sdpa_example(seed: int = 0, prompt_len: int = 1000, heads: int = 8, dim: int = 64):
    """q, k, v as ``[tokens, heads, dim]`` fp32.

    Drawn as one normal tensor of shape (3, 1, heads, prompt_len, dim) after
    seeding the global-style generator with ``seed`` (the glossary example's
    recipe), then moved to the token-major layout the library uses.
    """
    g = torch.Generator().manual_seed(int(seed))
    qkv = torch.randn(3, 1, heads, prompt_len, dim, generator=g)
    q, k, v = (t[0].permute(1, 0, 2).contiguous() for t in qkv.unbind(0))
    return q, k, v


def gqa_prompt(n_tokens: int, seed: int, hq: int = 32, hkv: int = 8, dim: int = 128,
               dtype=torch.bfloat16):
    """q ``[n, hq, dim]``, k/v ``[n, hkv, dim]`` iid N(0,1) in ``dtype``."""
    q = normal((n_tokens, hq, dim), seed * 3 + 0, dtype)
    k = normal((n_tokens, hkv, dim), seed * 3 + 1, dtype)
    v = normal((n_tokens, hkv, dim), seed * 3 + 2, dtype)
    return q, k, v


# Prompt lengths of the query-padding workload (each run twice).
LADDER_PROMPT_LENGTHS = (1041, 1468, 3118, 3788, 1137, 1200)


def ladder_prompt(idx: int, **kw):
    """The idx-th prompt of the query-padding workload (seed 10 + idx)."""
    return gqa_prompt(LADDER_PROMPT_LENGTHS[idx], 10 + idx, **kw)


def rolling_prompt(aligned_len: int, seed: int = 3, heads: int = 16, dim: int = 128,
                   dtype=torch.float16):
    """q, k, v ``[aligned_len, heads, dim]`` for the rolling-cache workload.

    Every position, including the left-pad positions, gets N(0,1) values; the
    pad positions are excluded by the mask, not by their contents.
    """
    return gqa_prompt(aligned_len, seed, hq=heads, hkv=heads, dim=dim, dtype=dtype)


@dataclass
class MixedBatch:
    """Inputs of the token-budget mixed-step workload (paged KV cache)."""

    page_size: int
    num_pages: int
    max_blocks: int
    decode_ctx: list          # context length of each running decode (keys incl. the new token)
    prompt_lens: list         # lengths of the waiting prompts
    block_table: torch.Tensor  # int32 [n_decode + n_prompt, max_blocks], -1 = unassigned
    seed: int


def mixed_batch(n_decode: int = 64, ctx_lo: int = 512, ctx_hi: int = 8192,
                n_prompt: int = 4, prompt_len: int = 20000, page_size: int = 16,
                decode_tail: int = 64, seed: int = 5) -> MixedBatch:
    """Integer layout of the mixed-step workload.

    Decode contexts are uniform integers in [ctx_lo, ctx_hi] (inclusive).  Each
    sequence gets enough pages for its full length plus ``decode_tail`` more
    tokens; page ids are a seeded permutation of the pool, so neighbouring
    logical pages are scattered over the pool.
    """
    g = torch.Generator().manual_seed(int(seed))
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (n_decode,), generator=g).tolist()
    prompts = [int(prompt_len)] * n_prompt
    lengths = list(ctx) + prompts
    need = [-(-(n + decode_tail) // page_size) for n in lengths]
    max_blocks = max(need)
    num_pages = sum(need)
    perm = torch.randperm(num_pages, generator=g)
    table = torch.full((len(lengths), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(need):
        table[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
    return MixedBatch(page_size, num_pages, max_blocks, ctx, prompts, table, seed)
