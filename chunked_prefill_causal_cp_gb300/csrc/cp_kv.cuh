// cp_kv.cuh -- where key j of a sequence lives and which query sees it.
// Shared by the SIMT fp32 kernel and the decode kernel (the tensor-core
// kernel applies the same rules per tile).
//
// Key indices: CONTIG / PAGED index keys by absolute position (j = a).
// ROLLING walks the physical slots j in [0, min(n, C)) and maps each to the
// absolute position it currently holds: a(j) = n-1 - ((n-1-j) mod C), where n
// is the number of positions written so far; position a lives in slot a mod C.
#pragma once

#include "cp_internal.h"

namespace cp {

struct SeqKeys {
  int n;       // positions written, including this call's rows
  int nkeys;   // key indices to walk
  int lo;      // lowest visible position (rolling: left pad), else 0
};

__device__ __forceinline__ int key_pos(const CacheView& c, const SeqKeys& k, int j) {
  if (c.kind != CP_CACHE_ROLLING) return j;
  return k.n - 1 - ((k.n - 1 - j) % c.capacity);
}

// Element offset of key index j of (sequence s, KV head g); -1 if the page
// table entry is out of range.
__device__ __forceinline__ long long key_offset(const CacheView& c, int hkv, int d, int s, int g, int j) {
  if (c.kind != CP_CACHE_PAGED) return ((long long)(s * hkv + g) * c.capacity + j) * d;
  const int blk = j / c.page_size;
  if (blk >= c.max_blocks) return -1;
  const int page = c.block_table[(long long)s * c.max_blocks + blk];
  if (page < 0 || page >= c.num_pages) return -1;
  return ((long long)(page * hkv + g) * c.page_size + j % c.page_size) * d;
}

// Key walk of sequence s whose queries end at absolute position last_pos.
__device__ __forceinline__ SeqKeys seq_keys(const AttnArgs& a, int s, int n, int last_pos) {
  SeqKeys k;
  k.n = n;
  if (a.cache.kind == CP_CACHE_ROLLING) {
    k.nkeys = n < a.cache.capacity ? n : a.cache.capacity;
    const int lp = a.left_pad ? a.left_pad[s] : 0;
    k.lo = lp > 0 ? lp : 0;
  } else {
    k.nkeys = last_pos + 1;
    k.lo = 0;
  }
  return k;
}

}  // namespace cp
