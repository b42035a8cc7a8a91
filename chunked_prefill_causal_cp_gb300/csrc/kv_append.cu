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

// Buckets of the work list's counting sort: 128 keys each; pairs that see
// more keys than the last bucket holds share it.
constexpr int kOrderBuckets = 4096;
constexpr int kAppendBlock = 256;

__device__ __forceinline__ int order_bucket(int keys) {
  return min(max((keys + 127) >> 7, 0), kOrderBuckets - 1);
}

// Exclusive prefix sum of v over the kAppendBlock threads; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kAppendBlock / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < kAppendBlock / 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kAppendBlock / 32) wsum[lane] = w;
  }
  __syncthreads();
  const int res = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
  *total = wsum[kAppendBlock / 32 - 1];
  __syncthreads();  // wsum may be reused
  return res;
}

// The tensor-core kernel's work list, heaviest pairs first (see AppendArgs):
// a histogram of the pairs' key counts, a descending exclusive scan of it, and
// a second pass that places each pair at its bucket's cursor.  The sequences
// go kAppendBlock at a time: a scan of their pair counts gives each pair an
// index, and each thread takes pairs by index.  Entries past pairs_bound (only
// from malformed row offsets) are dropped and reported.
__device__ void build_pair_order(const AppendArgs& a) {
  __shared__ int hist[kOrderBuckets];
  __shared__ int s_off[kAppendBlock + 1], s_r[kAppendBlock], s_p[kAppendBlock];
  __shared__ int wsum[kAppendBlock / 32];
  const int tid = threadIdx.x;
  const int ppt = a.pair_tokens;
  for (int b = tid; b < kOrderBuckets; b += kAppendBlock) hist[b] = 0;
  __syncthreads();
  int total = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int s0 = 0; s0 < a.rows.num_seqs; s0 += kAppendBlock) {
      const int s = s0 + tid;
      int r = 0, p = 0, np = 0;
      if (s < a.rows.num_seqs) {
        r = seq_rows(a.rows, s);
        p = a.past[s];
        if (r >= a.pair_min_rows && r > 0) np = min((r + ppt - 1) / ppt, a.pairs_bound);
      }
      int chunk = 0;
      const int off = block_exclusive_scan(np, wsum, &chunk);
      s_off[tid] = off;
      s_r[tid] = r;
      s_p[tid] = p;
      if (tid == 0) s_off[kAppendBlock] = chunk;
      __syncthreads();
      for (int i = tid; i < chunk; i += kAppendBlock) {
        int lo = 0, hi = kAppendBlock - 1;  // last j with s_off[j] <= i
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int k = i - s_off[lo];
        const int b = order_bucket(s_p[lo] + min((k + 1) * ppt, s_r[lo]));
        if (pass == 0) {
          atomicAdd(&hist[b], 1);
        } else {
          const int pos = atomicAdd(&hist[b], 1);
          if (pos < a.pairs_bound)
            a.pair_order[pos] = make_int2(s0 + lo, k * ppt);
          else if (a.status)
            atomicOr(a.status, CP_DEV_BOUNDS);
        }
      }
      __syncthreads();
    }
    if (pass == 0) {
      // Thread t owns the buckets that come t-th from the top, per at a time;
      // each bucket becomes the index of its first entry.
      constexpr int per = kOrderBuckets / kAppendBlock;
      const int top = kOrderBuckets - 1 - tid * per;
      int sum = 0;
#pragma unroll
      for (int i = 0; i < per; ++i) sum += hist[top - i];
      int before = block_exclusive_scan(sum, wsum, &total);
#pragma unroll
      for (int i = 0; i < per; ++i) {
        const int c = hist[top - i];
        hist[top - i] = before;
        before += c;
      }
      __syncthreads();
    }
  }
  for (int i = min(total, a.pairs_bound) + tid; i < a.pairs_bound; i += kAppendBlock) a.pair_order[i] = make_int2(-1, 0);
}

__global__ void __launch_bounds__(kAppendBlock) kv_append_kernel(const AppendArgs a, int rows_total) {
  pdl_launch_dependents();
  pdl_wait();
  if (a.pair_order && blockIdx.x == gridDim.x - 1) {  // the extra CTA
    build_pair_order(a);
    return;
  }
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
  const int block = kAppendBlock;
  const long long grid = (threads + block - 1) / block + (a.pair_order ? 1 : 0);
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
