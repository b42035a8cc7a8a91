// cp_internal.h -- argument blocks shared between the C-ABI layer
// (cp_api.cu) and the kernel translation units.  Plain data only; every
// pointer is a device pointer unless marked otherwise.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/cp_api.h"

namespace cp {

// Keys per split of the memory-bound decode path.  Fixed, so a row's result
// never depends on how many other rows share the launch.
constexpr int kDecodeSplit = 512;

// How query rows map onto sequences.
struct SeqRows {
  int num_seqs;
  int rows_uniform;      // > 0: sequence s owns rows [s*rows_uniform, (s+1)*rows_uniform)
  const int* cu_rows;    // else: sequence s owns rows [cu_rows[s], cu_rows[s+1])
};

__host__ __device__ inline int seq_row0(const SeqRows& r, int s) {
  return r.rows_uniform > 0 ? s * r.rows_uniform : r.cu_rows[s];
}
__host__ __device__ inline int seq_rows(const SeqRows& r, int s) {
  return r.rows_uniform > 0 ? r.rows_uniform : r.cu_rows[s + 1] - r.cu_rows[s];
}

// Where a sequence's K/V live.
struct CacheView {
  int kind;          // cp_cache_kind
  int capacity;      // CONTIG / ROLLING slots per (sequence, KV head)
  int page_size;     // PAGED
  int num_pages;     // PAGED
  int max_blocks;    // PAGED
  const int* block_table;  // PAGED [num_seqs, max_blocks]
};

// Arguments of the attention kernels (tensor-core, SIMT fp32, decode).
struct AttnArgs {
  int hq, hkv, d, group;   // group = hq / hkv query heads per KV head
  float scale_log2;        // softmax scale * log2(e)
  SeqRows rows;
  CacheView cache;
  const int* past;         // [num_seqs] positions cached before this call's rows
  const int* left_pad;     // ROLLING [num_seqs] or nullptr
  int max_ctx;             // host bound: past + rows <= max_ctx (checked in kernel)
  int min_rows;            // sequences with fewer rows are skipped (routed elsewhere)
  const void* q;           // [rows_total, hq, d]
  const void* k;           // cache / pool base (SIMT and decode kernels)
  const void* v;
  void* out;               // [rows_total, hq, d]
  float* part_o;           // decode split partials [num_seqs * dec_rows, hq, max_splits, d]
  float* part_ml;          // [num_seqs * dec_rows, hq, max_splits, 2] (max, sum) in log2 domain
  int max_splits;
  int dec_rows;            // rows per sequence on the split-KV path (1, or k with k * group <= 16)
  int* status;             // optional CP_DEV_* bits
  int kv_direct;           // tensor-core kernel: this call's new K/V rows may be read from
                           // k_new / v_new ([rows_total, hkv, d]) instead of the paged pool
  // If set, the lengths are advanced by commit_add once the attention has read
  // them: by CTA (0, 0) right after the dependency wait when `past` is a copy
  // (it must not alias commit_lens; tensor-core, fp32 and split-KV kernels),
  // else through the ticket (tensor-core and fp32 kernels).
  int* commit_lens = nullptr;
  int commit_add = 0;
  unsigned* ticket = nullptr;  // the ticket counter (zero before the launch, left zero)
  // Tensor-core kernel, contiguous cache, fused append: the tiles that hold this
  // call's keys are read from k_new / v_new [num_seqs, rows_uniform, hkv, d] and
  // the kernel copies those rows into the cache [num_seqs, hkv, capacity, d].
  int fused = 0;
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  void* k_cache = nullptr;
  void* v_cache = nullptr;
  // Tensor-core kernel, ragged rows: if set, the work of cluster L (linear
  // index over the grid) is pair_order[L / hkv] for KV head L % hkv, a list the
  // append kernel wrote with the pairs that see the most keys first (entries
  // with a negative sequence are empty).  Else pair blockIdx.x / 2 of KV head
  // blockIdx.y, found by scanning the sequences.
  const int2* pair_order = nullptr;
};

struct AppendArgs {
  int hkv, d, esize;       // esize: bytes per element
  SeqRows rows;
  CacheView cache;
  const int* past;
  int max_ctx;
  const void* k_new;       // [rows_total, hkv, d]
  const void* v_new;
  void* k_cache;
  void* v_cache;
  int* status;
  int* past_snapshot = nullptr;  // optional [num_seqs]: CTA 0 copies past[] here
  // Optional work list for the tensor-core kernel that follows (ragged rows):
  // one extra CTA writes pairs_bound entries (sequence, first token) -- every
  // pair of pair_tokens tokens of the sequences with at least pair_min_rows
  // rows, ordered by the keys the pair's last token sees, most first (equal
  // counts in any order), then (-1, 0) entries up to pairs_bound.
  int2* pair_order = nullptr;
  int pair_tokens = 0;
  int pair_min_rows = 0;
  int pairs_bound = 0;
};

// Launches `kernel` with programmatic dependent launch allowed: the grid may
// be scheduled while the previous kernel in the stream is still running.
// Every kernel of this library triggers its dependents on entry and waits
// for the previous grid (griddepcontrol.wait) before it touches global
// memory, so only set-up that reads no global memory (barrier init, TMEM
// allocation) overlaps the previous kernel's tail.
#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Device side of programmatic dependent launch.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// ---- launchers (return cudaGetLastError() after the launch) ----
cudaError_t launch_kv_append(const AppendArgs& a, int rows_total, cudaStream_t st);
// status (optional): CP_DEV_BOUNDS is set for a sequence with no rows.
cudaError_t launch_commit(int* lens, const SeqRows& rows, int add_uniform, int* status, cudaStream_t st);
// Widens up to three tensors (null entries skipped) in one launch.
cudaError_t launch_pad_rows(void* const base[3], const int row_bytes[3], int batch, int rows_padded, int real_rows,
                            cudaStream_t st);
cudaError_t launch_attn_f32(const AttnArgs& a, int rows_bound, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnArgs& a, int dtype, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const CUtensorMap& tkn,
                           const CUtensorMap& tvn, int pairs_bound, cudaStream_t st);
// Split-KV decode: partials into a.part_o / a.part_ml, then their combine.  Takes the
// sequences with exactly a.dec_rows rows (a.dec_rows * a.group <= 16).
cudaError_t launch_decode(const AttnArgs& a, int dtype, cudaStream_t st);
// Most rows per sequence the split-KV path takes for a GQA group of `group` heads.
constexpr int decode_max_rows(int group) { return group > 0 ? 16 / group : 0; }

// Every check cp_mixed_step makes before enqueueing anything (returns its
// status); *ws_need is the workspace the step then needs (decode partials).
int mixed_step_check(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new,
                     const void* k_pages, const void* v_pages, const int32_t* block_table, const int32_t* cu_rows,
                     const int32_t* past_len, int32_t num_seqs, int32_t total_rows, int32_t max_ctx, const void* out,
                     size_t* ws_need);

// Tensor-core path tiling (shared with the host so it can size grids and
// tensor-map boxes).
constexpr int kTcBlockM = 128;   // packed (token, head) rows per CTA
constexpr int kTcBlockN = 128;   // keys per KV tile
bool attn_tc_supported(int d, int group, int dtype);
bool decode_supported(int d, int group, int dtype);

}  // namespace cp
