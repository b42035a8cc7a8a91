// kv_append.cu -- the KV append kernel and the seqlens commit kernel.
//
// Append ([Wiki] 一.1, [Horizon] 3, [Glossary] PagedAttention): each new K/V
// row of D elements is copied to the slot of its absolute position with
// 16-byte vector loads/stores; a bit-exact copy, nothing else in the cache is
// touched.  One group of D*esize/16 threads moves one (token, KV head) row of
// K and the same row of V.
//
// Commit ([Wiki] 四, rewind to past + real rows): lens[s] += rows.
#include <cstdint>

#include "cp_internal.h"

namespace cp {
namespace {

__device__ __forceinline__ int find_seq(const SeqRows& r, int row) {
  if (r.rows_uniform > 0) return row / r.rows_uniform;
  int lo = 0, hi = r.num_seqs - 1;  // last s with cu_rows[s] <= row
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (r.cu_rows[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Destination element offset of (sequence s, KV head g, absolute position pos),
// or -1 when the position is outside the cache the host bounds allow.
__device__ __forceinline__ long long slot_offset(const CacheView& c, int hkv, int d, int s, int g, int pos,
                                                 int max_ctx) {
  if (pos < 0 || pos >= max_ctx) return -1;
  if (c.kind == CP_CACHE_CONTIG) {
    if (pos >= c.capacity) return -1;
    return ((long long)(s * hkv + g) * c.capacity + pos) * d;
  }
  if (c.kind == CP_CACHE_ROLLING) {
    return ((long long)(s * hkv + g) * c.capacity + pos % c.capacity) * d;
  }
  const int blk = pos / c.page_size;
  if (blk >= c.max_blocks) return -1;
  const int page = c.block_table[(long long)s * c.max_blocks + blk];
  if (page < 0 || page >= c.num_pages) return -1;
  return ((long long)(page * hkv + g) * c.page_size + pos % c.page_size) * d;
}

__global__ void kv_append_kernel(const AppendArgs a, int rows_total) {
  pdl_launch_dependents();
  pdl_wait();
  if (a.past_snapshot && blockIdx.x == 0)
    for (int s = threadIdx.x; s < a.rows.num_seqs; s += blockDim.x) a.past_snapshot[s] = a.past[s];
  const int vec_per_row = a.d * a.esize / 16;           // 16-byte vectors per row
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid / vec_per_row;              // (token, head) row
  const int lane_vec = (int)(gid % vec_per_row);
  if (row >= (long long)rows_total * a.hkv) return;
  const int t = (int)(row / a.hkv);
  const int g = (int)(row % a.hkv);
  const int s = find_seq(a.rows, t);
  const int pos = a.past[s] + (t - seq_row0(a.rows, s));
  const long long dst = slot_offset(a.cache, a.hkv, a.d, s, g, pos, a.max_ctx);
  if (dst < 0) {
    if (a.status && lane_vec == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const long long src_b = (row * a.d) * a.esize + (long long)lane_vec * 16;
  const long long dst_b = dst * a.esize + (long long)lane_vec * 16;
  const uint4 kv = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_new) + src_b);
  const uint4 vv = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_new) + src_b);
  *reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + dst_b) = kv;
  *reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + dst_b) = vv;
}

// Rows [real_rows, rows_padded) of each sequence become copies of row
// real_rows - 1 ([Wiki] 四: pad rows repeat the last real token).  One launch
// widens up to three tensors: blockIdx.y picks the tensor (a null one is skipped).
struct PadTensors {
  char* base[3];
  int row_bytes[3];
};

__global__ void pad_rows_kernel(const PadTensors p, int batch, int rows_padded, int real_rows) {
  pdl_launch_dependents();
  pdl_wait();
  char* base = p.base[blockIdx.y];
  const int row_bytes = p.row_bytes[blockIdx.y];
  if (base == nullptr) return;
  const int vecs = row_bytes / 16;
  const int pad = rows_padded - real_rows;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)batch * pad * vecs) return;
  const int vec = (int)(gid % vecs);
  const long long r = gid / vecs;
  const int b = (int)(r / pad);
  const int t = real_rows + (int)(r % pad);
  const char* src = base + ((long long)b * rows_padded + real_rows - 1) * row_bytes;
  char* dst = base + ((long long)b * rows_padded + t) * row_bytes;
  reinterpret_cast<uint4*>(dst)[vec] = reinterpret_cast<const uint4*>(src)[vec];
}

// Advances each sequence's length by its rows (or by add_uniform); with
// `status`, a sequence with no rows is reported (a mixed step lists only
// sequences that have rows in it).
__global__ void commit_kernel(int* lens, const SeqRows rows, int add_uniform, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= rows.num_seqs) return;
  const int r = add_uniform >= 0 ? add_uniform : seq_rows(rows, s);
  if (status && r < 1) atomicOr(status, CP_DEV_BOUNDS);
  lens[s] += r;
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, int rows_total, cudaStream_t st) {
  const long long vec_per_row = a.d * a.esize / 16;
  const long long threads = (long long)rows_total * a.hkv * vec_per_row;
  if (threads == 0) return cudaSuccess;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  return launch_pdl(kv_append_kernel, dim3((unsigned)grid), dim3(block), 0, st, a, rows_total);
}

cudaError_t launch_pad_rows(void* const base[3], const int row_bytes[3], int batch, int rows_padded, int real_rows,
                            cudaStream_t st) {
  PadTensors p;
  long long threads = 0;
  for (int i = 0; i < 3; ++i) {
    p.base[i] = static_cast<char*>(base[i]);
    p.row_bytes[i] = row_bytes[i];
    const long long t = base[i] ? (long long)batch * (rows_padded - real_rows) * (row_bytes[i] / 16) : 0;
    if (t > threads) threads = t;
  }
  if (threads <= 0) return cudaSuccess;
  const int block = 256;
  return launch_pdl(pad_rows_kernel, dim3((unsigned)((threads + block - 1) / block), 3), dim3(block), 0, st, p,
                    batch, rows_padded, real_rows);
}

// add_uniform >= 0 adds that count to every sequence; -1 adds each
// sequence's own row count.
cudaError_t launch_commit(int* lens, const SeqRows& rows, int add_uniform, int* status, cudaStream_t st) {
  if (rows.num_seqs == 0) return cudaSuccess;
  const int block = 128;
  return launch_pdl(commit_kernel, dim3((rows.num_seqs + block - 1) / block), dim3(block), 0, st, lens, rows,
                    add_uniform, status);
}

}  // namespace cp
