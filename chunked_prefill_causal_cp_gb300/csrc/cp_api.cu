// cp_api.cu -- the C ABI: argument checks, tensor-map setup and the launches
// behind cp_kv_append, cp_prefill_chunk_attn, cp_mixed_step and
// cp_workspace_size.  Every argument is checked before anything is enqueued.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "cp_internal.h"

using namespace cp;

namespace {

int esize_of(int dtype) { return dtype == CP_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_desc(const cp_layer_desc* d, bool need_batch) {
  if (d == nullptr) return CP_ERR_INVALID_ARG;
  if (d->dtype != CP_F32 && d->dtype != CP_BF16 && d->dtype != CP_F16) return CP_ERR_INVALID_ARG;
  if (need_batch && d->batch <= 0) return CP_ERR_INVALID_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0) return CP_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return CP_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return CP_ERR_UNSUPPORTED;
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return CP_ERR_INVALID_ARG;
  switch (d->kind) {
    case CP_CACHE_CONTIG:
    case CP_CACHE_ROLLING:
      if (d->capacity <= 0) return CP_ERR_INVALID_ARG;
      break;
    case CP_CACHE_PAGED:
      if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64 && d->page_size != 128)
        return CP_ERR_UNSUPPORTED;
      if (d->num_pages <= 0 || d->max_blocks <= 0) return CP_ERR_INVALID_ARG;
      break;
    default:
      return CP_ERR_INVALID_ARG;
  }
  return CP_OK;
}

// Upper bound of positions a sequence may reach in this layout.
int64_t layout_limit(const cp_layer_desc* d) {
  if (d->kind == CP_CACHE_CONTIG) return d->capacity;
  if (d->kind == CP_CACHE_PAGED) return (int64_t)d->max_blocks * d->page_size;
  return INT32_MAX;  // rolling: positions grow without bound, slots wrap
}

CacheView make_cache(const cp_layer_desc* d, const int32_t* block_table) {
  CacheView c;
  c.kind = d->kind;
  c.capacity = d->capacity;
  c.page_size = d->page_size;
  c.num_pages = d->num_pages;
  c.max_blocks = d->max_blocks;
  c.block_table = block_table;
  return c;
}

float scale_log2(const cp_layer_desc* d) {
  const double sc = d->scale > 0.f ? (double)d->scale : 1.0 / std::sqrt((double)d->head_dim);
  return (float)(sc * 1.4426950408889634);  // log2(e)
}

int64_t max_splits_for(int32_t max_ctx) { return ((int64_t)max_ctx + kDecodeSplit - 1) / kDecodeSplit; }

// Workspace of cp_prefill_chunk: a 256-byte control block (the fused
// kernel's ticket counter, zero between calls), then a copy of seqlens_k in
// whole 256-byte blocks, then the split partials.  The other calls use the
// partials only, from the start of the workspace.
constexpr int64_t kControlBytes = 256;
int64_t snapshot_bytes(int32_t num_seqs) { return ((int64_t)num_seqs * 4 + 255) / 256 * 256; }

// Decode workspace: the split partials (output rows, then max and sum) of
// `rows` query rows on the split-KV path.
int64_t decode_ws_bytes(const cp_layer_desc* d, int32_t max_ctx, int64_t rows) {
  const int64_t ms = max_splits_for(max_ctx);
  return rows * d->num_q_heads * ms * (d->head_dim + 2) * (int64_t)sizeof(float);
}

// Rows per sequence a call with `rows_uniform` rows each puts on the split-KV
// path: all of them when rows_uniform * G <= 16 (a decode row, or a short chunk
// such as k verified draft tokens), else only one-row sequences (1).
int decode_rows_for(const cp_layer_desc* d, int rows_uniform) {
  const int G = d->num_q_heads / d->num_kv_heads;
  return rows_uniform >= 1 && rows_uniform <= decode_max_rows(G) ? rows_uniform : 1;
}

// ---- tensor maps (driver entry point fetched through the runtime)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D tensor of 16-bit elements: dims {d0 (contiguous), d1, d2}, 128-byte
// swizzled boxes; out-of-range box elements read as zero.
bool encode_3d(CUtensorMap* m, int dtype, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty =
      dtype == CP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D tensor of 16-bit elements {d0 (contiguous), d1, d2, d3}, 128-byte swizzled boxes.
bool encode_4d(CUtensorMap* m, int dtype, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
               uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      dtype == CP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Page-row map of a [rows, 128] 16-bit pool (rows a multiple of 8): the 4-D
// view {64 columns, 8 rows (256 B apart), 2 halves (128 B apart), rows / 8
// groups (2048 B apart)} with one page per box, so a box lands as
// [page / 8][half][8 rows][128 B] (128-byte swizzle).
bool encode_page_rows(CUtensorMap* m, int dtype, const void* base, uint64_t rows, uint32_t page) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 8 || page % 8 || page / 8 > 256) return false;
  const cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  const cuuint64_t strides[3] = {256, 128, 2048};
  const cuuint32_t box[4] = {64, 8, 2, page / 8};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      dtype == CP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the tensor-core path: Q/out rows [rows_total, Hq, D] in
// boxes of (64 dims, G heads, 128/G tokens); K/V in boxes of 128 keys
// (contiguous / rolling) or one page (paged) by 64 dims, or on a paged cache
// with D = 128 page-row maps (one box per page, both halves).
bool make_tc_maps(const cp_layer_desc* d, const void* q, const void* out, int64_t rows_total, const void* k,
                  const void* v, int batch, CUtensorMap* tq, CUtensorMap* to, CUtensorMap* tk, CUtensorMap* tv) {
  const int G = d->num_q_heads / d->num_kv_heads;
  const uint64_t D = d->head_dim;
  if (!encode_3d(tq, d->dtype, q, D, d->num_q_heads, (uint64_t)rows_total, 64, G, kTcBlockM / G)) return false;
  if (!encode_3d(to, d->dtype, out, D, d->num_q_heads, (uint64_t)rows_total, 64, G, kTcBlockM / G)) return false;
  if (d->kind == CP_CACHE_PAGED) {
    const uint64_t planes = (uint64_t)d->num_pages * d->num_kv_heads;
    if (D == 128)
      return encode_page_rows(tk, d->dtype, k, planes * d->page_size, d->page_size) &&
             encode_page_rows(tv, d->dtype, v, planes * d->page_size, d->page_size);
    return encode_3d(tk, d->dtype, k, D, d->page_size, planes, 64, d->page_size, 1) &&
           encode_3d(tv, d->dtype, v, D, d->page_size, planes, 64, d->page_size, 1);
  }
  const uint64_t planes = (uint64_t)batch * d->num_kv_heads;
  return encode_3d(tk, d->dtype, k, D, d->capacity, planes, 64, kTcBlockN, 1) &&
         encode_3d(tv, d->dtype, v, D, d->capacity, planes, 64, kTcBlockN, 1);
}

int launch_result(cudaError_t e) { return e == cudaSuccess ? CP_OK : CP_ERR_CUDA; }

int run_tc_part(const cp_layer_desc* d, AttnArgs a, int64_t rows_total, const void* k, const void* v,
                int batch_for_maps, cudaStream_t st, const void* k_new, const void* v_new, bool decode_ok, int kdec);

// A caller-provided side stream and two events: when a call launches both the
// split-KV kernels and the tensor-core kernel, the split-KV ones run on `side`
// (forked from `st` after what came before, joined back before what follows),
// so the memory-bound and the tensor-bound work share the GPU.
struct ForkJoin {
  cudaStream_t side;
  cudaEvent_t fork, join;
};

// Attention over every sequence of `rows`, routed by dtype and row count.
// k_new / v_new (may be NULL): this call's new K/V rows [rows_total, Hkv, D]; when given with a
// paged cache, the tensor-core kernel reads the tiles made only of new rows from them.
// fj (may be NULL): run the split-KV part beside the tensor-core part, as above.
int run_attention(const cp_layer_desc* d, const AttnArgs& base, int64_t rows_total, int rows_max_per_seq,
                  const void* k, const void* v, int batch_for_maps, void* workspace, size_t ws_bytes,
                  cudaStream_t st, const void* k_new = nullptr, const void* v_new = nullptr,
                  const ForkJoin* fj = nullptr) {
  const int G = d->num_q_heads / d->num_kv_heads;
  AttnArgs a = base;
  if (d->dtype == CP_F32) {
    a.min_rows = 1;
    return launch_result(launch_attn_f32(a, rows_max_per_seq, st));
  }
  const bool decode_ok = decode_supported(d->head_dim, G, d->dtype) && d->kind != CP_CACHE_ROLLING;
  if (!attn_tc_supported(d->head_dim, G, d->dtype)) return CP_ERR_UNSUPPORTED;
  // Uniform rows of at most 16 / G per sequence all take the split-KV path;
  // otherwise it takes the one-row sequences and the tensor-core kernel the rest.
  const int kdec = decode_rows_for(d, base.rows.rows_uniform);
  const bool any_multi = rows_max_per_seq > kdec;
  const bool any_single = base.rows.rows_uniform == 0 || base.rows.rows_uniform == kdec;
  const bool run_dec = decode_ok && any_single, run_tc = any_multi || !decode_ok;
  const bool forked = fj != nullptr && run_dec && run_tc;
  if (run_dec) {
    const int64_t need = decode_ws_bytes(d, a.max_ctx, (int64_t)a.rows.num_seqs * kdec);
    if (workspace == nullptr || (int64_t)ws_bytes < need) return CP_ERR_WORKSPACE;
    AttnArgs dec = a;
    dec.dec_rows = kdec;
    if (run_tc) dec.commit_lens = nullptr;  // the tensor-core kernel advances the lengths
    dec.part_o = static_cast<float*>(workspace);
    dec.max_splits = (int)max_splits_for(a.max_ctx);
    dec.part_ml =
        dec.part_o + (int64_t)a.rows.num_seqs * kdec * d->num_q_heads * dec.max_splits * d->head_dim;
    cudaStream_t dst = st;
    if (forked) {
      if (cudaEventRecord(fj->fork, st) != cudaSuccess || cudaStreamWaitEvent(fj->side, fj->fork, 0) != cudaSuccess)
        return CP_ERR_CUDA;
      dst = fj->side;
    }
    int r = launch_result(launch_decode(dec, d->dtype, dst));
    if (forked && cudaEventRecord(fj->join, fj->side) != cudaSuccess && r == CP_OK) r = CP_ERR_CUDA;
    if (r != CP_OK) {
      if (forked) cudaStreamWaitEvent(st, fj->join, 0);
      return r;
    }
  }
  if (run_tc) {
    const int r = run_tc_part(d, a, rows_total, k, v, batch_for_maps, st, k_new, v_new, decode_ok, kdec);
    if (forked && cudaStreamWaitEvent(st, fj->join, 0) != cudaSuccess && r == CP_OK) return CP_ERR_CUDA;
    return r;
  }
  return CP_OK;
}

// The tensor-core part of run_attention.
int run_tc_part(const cp_layer_desc* d, AttnArgs a, int64_t rows_total, const void* k, const void* v,
                int batch_for_maps, cudaStream_t st, const void* k_new, const void* v_new, bool decode_ok, int kdec) {
  const int G = d->num_q_heads / d->num_kv_heads;
  a.min_rows = decode_ok ? kdec + 1 : 1;
  CUtensorMap tq, to, tk, tv, tkn, tvn;
  if (!make_tc_maps(d, a.q, a.out, rows_total, k, v, batch_for_maps, &tq, &to, &tk, &tv)) return CP_ERR_CUDA;
  std::memset(&tkn, 0, sizeof(tkn));
  std::memset(&tvn, 0, sizeof(tvn));
  a.kv_direct = 0;
  if (d->kind == CP_CACHE_PAGED && k_new && v_new) {
    const uint64_t D = d->head_dim;
    if (!encode_3d(&tkn, d->dtype, k_new, D, d->num_kv_heads, (uint64_t)rows_total, 64, 1, kTcBlockN) ||
        !encode_3d(&tvn, d->dtype, v_new, D, d->num_kv_heads, (uint64_t)rows_total, 64, 1, kTcBlockN))
      return CP_ERR_CUDA;
    a.kv_direct = 1;
  }
  const int ppt = 2 * (kTcBlockM / G);  // tokens per pair of 128-row Q tiles
  int64_t pairs;
  if (a.rows.rows_uniform > 0)
    pairs = (int64_t)a.rows.num_seqs * ((a.rows.rows_uniform + ppt - 1) / ppt);
  else
    pairs = (rows_total + ppt - 1) / ppt + a.rows.num_seqs;
  if (2 * pairs > INT32_MAX) return CP_ERR_UNSUPPORTED;
  return launch_result(launch_attn_tc(a, d->dtype, tq, tk, tv, to, tkn, tvn, (int)pairs, st));
}

// A chunk of uniform rows in half precision goes to the tensor-core kernel
// with the append fused in: on a contiguous cache when it has more rows than
// the split-KV path takes; on a ring wider than one tile when rows <= capacity
// - 128 (the geometry in which the kernel walks a ring's cached and new slots
// apart, as it then also does for an unfused ring call).
bool use_fused(const cp_layer_desc* d, int32_t rows_padded) {
  const int G = d->num_q_heads / d->num_kv_heads;
  if (d->dtype == CP_F32 || !attn_tc_supported(d->head_dim, G, d->dtype)) return false;
  if (d->kind == CP_CACHE_ROLLING) return d->capacity > kTcBlockN && rows_padded <= d->capacity - kTcBlockN;
  const bool on_decode_path = decode_supported(d->head_dim, G, d->dtype) && rows_padded <= decode_max_rows(G);
  return d->kind == CP_CACHE_CONTIG && rows_padded > 1 && !on_decode_path;
}

// One launch for append, attention and the advance of the lengths: the tiles
// that hold the chunk's keys are read from k_new / v_new (4-D maps over
// [batch, rows_padded, Hkv, D]), the kernel copies those rows into the cache,
// and the last CTA to take a ticket adds a.commit_add to a.commit_lens.
int run_fused(const cp_layer_desc* d, AttnArgs a, int64_t rows_total, const void* k_new, const void* v_new,
              cudaStream_t st) {
  const int G = d->num_q_heads / d->num_kv_heads;
  const uint64_t D = d->head_dim;
  const int rows_padded = a.rows.rows_uniform;
  CUtensorMap tq, to, tk, tv, tkn, tvn;
  if (!make_tc_maps(d, a.q, a.out, rows_total, a.k, a.v, d->batch, &tq, &to, &tk, &tv) ||
      !encode_4d(&tkn, d->dtype, k_new, D, d->num_kv_heads, rows_padded, d->batch, 64, 1, kTcBlockN, 1) ||
      !encode_4d(&tvn, d->dtype, v_new, D, d->num_kv_heads, rows_padded, d->batch, 64, 1, kTcBlockN, 1))
    return CP_ERR_CUDA;
  a.min_rows = 1;
  a.kv_direct = 0;
  a.fused = 1;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = const_cast<void*>(a.k);
  a.v_cache = const_cast<void*>(a.v);
  const int ppt = 2 * (kTcBlockM / G);
  const int64_t pairs = (int64_t)d->batch * ((rows_padded + ppt - 1) / ppt);
  if (2 * pairs > INT32_MAX) return CP_ERR_UNSUPPORTED;
  return launch_result(launch_attn_tc(a, d->dtype, tq, tk, tv, to, tkn, tvn, (int)pairs, st));
}

// Append, attention and length advance of a step whose sequences have
// ragged rows (cu_rows): every row's K/V is appended first (pages through the
// block table, or the contiguous cache when block_table is NULL), then
// one-row sequences take the split-KV decode path and the others the
// tensor-core path, reading the lengths as they were before the step; a last
// kernel advances each length by its own rows.  Arguments already checked.
// Where a ragged call's work list goes: after the split-KV partials, 16-byte
// aligned, one int2 per pair the tensor-core grid has room for.  `use` is false
// when the tensor-core kernel will not run (fp32 layers, or one row per
// sequence on the split-KV path).
struct PairOrderPlan {
  bool use;
  int64_t offset, bytes;
  int pair_tokens, min_rows, pairs_bound;
};

PairOrderPlan pair_order_plan(const cp_layer_desc* d, int64_t total_rows, int32_t max_ctx, int32_t num_seqs,
                              int64_t max_rows_per_seq) {
  PairOrderPlan p{false, 0, 0, 0, 0, 0};
  const int G = d->num_q_heads / d->num_kv_heads;
  if (d->dtype == CP_F32 || !attn_tc_supported(d->head_dim, G, d->dtype)) return p;
  const bool decode_ok = decode_supported(d->head_dim, G, d->dtype) && d->kind != CP_CACHE_ROLLING;
  const int kdec = decode_rows_for(d, 0);
  if (decode_ok && max_rows_per_seq <= kdec) return p;
  const int64_t dec_need = decode_ok ? decode_ws_bytes(d, max_ctx, num_seqs) : 0;
  const int ppt = 2 * (kTcBlockM / G);
  const int64_t pairs = (total_rows + ppt - 1) / ppt + num_seqs;  // the tensor-core grid's pair bound
  if (2 * pairs > INT32_MAX) return p;
  p.use = true;
  p.offset = (dec_need + 15) / 16 * 16;
  p.bytes = pairs * 8;
  p.pair_tokens = ppt;
  p.min_rows = decode_ok ? kdec + 1 : 1;
  p.pairs_bound = (int)pairs;
  return p;
}

int ragged_step(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new, void* k_cache,
                void* v_cache, const int32_t* block_table, const int32_t* cu_rows, int32_t* past_len,
                int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, cudaStream_t st, const ForkJoin* fj = nullptr) {
  const SeqRows rows{num_seqs, 0, cu_rows};
  const CacheView cache = make_cache(desc, block_table);

  AppendArgs ap;
  ap.hkv = desc->num_kv_heads;
  ap.d = desc->head_dim;
  ap.esize = esize_of(desc->dtype);
  ap.rows = rows;
  ap.cache = cache;
  ap.past = past_len;
  ap.max_ctx = max_ctx;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_cache = k_cache;
  ap.v_cache = v_cache;
  ap.status = dev_status;
  // Every listed sequence has at least one row, so none has more than
  // total_rows - num_seqs + 1; with one row each the tensor-core path has no
  // work and is not launched.
  const int64_t max_rows_per_seq = total_rows >= num_seqs ? (int64_t)total_rows - num_seqs + 1 : total_rows;
  // The tensor-core kernel's heaviest-first work list, built by the append
  // kernel, when the workspace has room for it after the split-KV partials.
  const PairOrderPlan plan = pair_order_plan(desc, total_rows, max_ctx, num_seqs, max_rows_per_seq);
  if (plan.use && workspace && aligned16(workspace) && (int64_t)workspace_bytes >= plan.offset + plan.bytes) {
    ap.pair_order = reinterpret_cast<int2*>(static_cast<char*>(workspace) + plan.offset);
    ap.pair_tokens = plan.pair_tokens;
    ap.pair_min_rows = plan.min_rows;
    ap.pairs_bound = plan.pairs_bound;
  }
  int r = launch_result(launch_kv_append(ap, total_rows, st));
  if (r != CP_OK) return r;

  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.hq = desc->num_q_heads;
  a.hkv = desc->num_kv_heads;
  a.d = desc->head_dim;
  a.group = a.hq / a.hkv;
  a.scale_log2 = scale_log2(desc);
  a.rows = rows;
  a.cache = cache;
  a.past = past_len;
  a.max_ctx = max_ctx;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.status = dev_status;
  a.pair_order = ap.pair_order;
  const bool paged = desc->kind == CP_CACHE_PAGED;
  r = run_attention(desc, a, total_rows, (int)max_rows_per_seq, k_cache, v_cache, paged ? 0 : desc->batch, workspace,
                    workspace_bytes, st, paged ? k_new : nullptr, paged ? v_new : nullptr, fj);
  if (r != CP_OK) return r;
  return launch_result(launch_commit(past_len, rows, -1, dev_status, st));
}

}  // namespace

namespace cp {

// Every check cp_mixed_step makes before it enqueues anything; *ws_need is the
// workspace it then needs (the decode rows' split-KV partials; 0 when the
// layer takes no decode path).  Returns CP_OK or the status cp_mixed_step
// returns.
int mixed_step_check(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new,
                     const void* k_pages, const void* v_pages, const int32_t* block_table, const int32_t* cu_rows,
                     const int32_t* past_len, int32_t num_seqs, int32_t total_rows, int32_t max_ctx, const void* out,
                     size_t* ws_need) {
  *ws_need = 0;
  int r = check_desc(desc, false);
  if (r != CP_OK) return r;
  if (desc->kind != CP_CACHE_PAGED) return CP_ERR_UNSUPPORTED;
  if (num_seqs <= 0 || total_rows < 0 || max_ctx <= 0) return CP_ERR_INVALID_ARG;
  if (total_rows == 0) return CP_OK;
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !block_table || !cu_rows || !past_len || !out)
    return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(out))
    return CP_ERR_INVALID_ARG;
  if ((int64_t)max_ctx > layout_limit(desc)) return CP_ERR_CAPACITY;
  // Checks the attention launches would make, taken before the append is enqueued.
  const int G0 = desc->num_q_heads / desc->num_kv_heads;
  if (desc->dtype != CP_F32) {
    if (!attn_tc_supported(desc->head_dim, G0, desc->dtype)) return CP_ERR_UNSUPPORTED;
    if (decode_supported(desc->head_dim, G0, desc->dtype)) *ws_need = (size_t)decode_ws_bytes(desc, max_ctx, num_seqs);
  }
  return CP_OK;
}

}  // namespace cp

extern "C" {

size_t cp_workspace_size(const cp_layer_desc* desc, int32_t max_rows, int32_t max_ctx, int32_t num_seqs) {
  if (check_desc(desc, false) != CP_OK || max_rows < 0 || max_ctx < 0 || num_seqs < 0) return 0;
  // Split-KV partials: for each sequence, as many rows as a call of at most
  // max_rows rows can put on the split-KV path (1, or up to 16 / G rows).
  int64_t dec_rows = num_seqs;
  if (num_seqs > 0) {
    const int G = desc->num_q_heads / desc->num_kv_heads;
    const int64_t per_seq = std::max<int64_t>(1, ((int64_t)max_rows + num_seqs - 1) / num_seqs);
    dec_rows = (int64_t)num_seqs * std::min<int64_t>(per_seq, decode_max_rows(G));
  }
  // A ragged call's work list for the tensor-core kernel (one int2 per pair),
  // placed after its split-KV partials (which the terms above cover).
  int64_t order = 0;
  const int G = desc->num_q_heads / desc->num_kv_heads;
  if (desc->dtype != CP_F32 && attn_tc_supported(desc->head_dim, G, desc->dtype)) {
    const int ppt = 2 * (kTcBlockM / G);
    order = ((int64_t)(max_rows + ppt - 1) / ppt + num_seqs) * 8 + 16;
  }
  return (size_t)(kControlBytes + snapshot_bytes(num_seqs) + decode_ws_bytes(desc, max_ctx, dec_rows) + order);
}

int cp_kv_append(const cp_layer_desc* desc, const void* k_new, const void* v_new, int32_t rows, void* k_cache,
                 void* v_cache, const int32_t* seqlens_k, const int32_t* block_table, int32_t max_past,
                 int32_t* dev_status, void* stream) {
  int r = check_desc(desc, true);
  if (r != CP_OK) return r;
  if (rows < 0 || max_past < 0) return CP_ERR_INVALID_ARG;
  if (rows == 0) return CP_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !seqlens_k) return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_PAGED && !block_table) return CP_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_ROLLING) {
    if (rows > desc->capacity) return CP_ERR_CAPACITY;
  } else if ((int64_t)max_past + rows > layout_limit(desc)) {
    return CP_ERR_CAPACITY;
  }
  if ((int64_t)desc->batch * rows > INT32_MAX) return CP_ERR_UNSUPPORTED;
  AppendArgs a;
  a.hkv = desc->num_kv_heads;
  a.d = desc->head_dim;
  a.esize = esize_of(desc->dtype);
  a.rows = SeqRows{desc->batch, rows, nullptr};
  a.cache = make_cache(desc, block_table);
  a.past = seqlens_k;
  a.max_ctx = (int)std::min<int64_t>((int64_t)max_past + rows, INT32_MAX);
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.status = dev_status;
  return launch_result(launch_kv_append(a, desc->batch * rows, static_cast<cudaStream_t>(stream)));
}

int cp_pad_chunk(const cp_layer_desc* desc, void* q, void* k_new, void* v_new, int32_t real_rows,
                 int32_t rows_padded, void* stream) {
  int r = check_desc(desc, true);
  if (r != CP_OK) return r;
  if (real_rows <= 0 || rows_padded < real_rows) return CP_ERR_INVALID_ARG;
  if ((q && !aligned16(q)) || (k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new))) return CP_ERR_INVALID_ARG;
  if ((int64_t)desc->batch * rows_padded > INT32_MAX) return CP_ERR_UNSUPPORTED;
  if (rows_padded == real_rows) return CP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int es = esize_of(desc->dtype);
  const int qb = desc->num_q_heads * desc->head_dim * es;
  const int kb = desc->num_kv_heads * desc->head_dim * es;
  void* const base[3] = {q, k_new, v_new};
  const int row_bytes[3] = {qb, kb, kb};
  return launch_result(launch_pad_rows(base, row_bytes, desc->batch, rows_padded, real_rows, st));
}

int cp_prefill_chunk_attn(const cp_layer_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                          int32_t* seqlens_k, const int32_t* block_table, const int32_t* left_pad,
                          int32_t rows_padded, int32_t real_rows, int32_t max_past, void* out, void* workspace,
                          size_t workspace_bytes, int32_t commit, int32_t* dev_status, void* stream) {
  int r = check_desc(desc, true);
  if (r != CP_OK) return r;
  if (rows_padded <= 0 || real_rows <= 0 || real_rows > rows_padded || max_past < 0) return CP_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !seqlens_k || !out) return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_PAGED && !block_table) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_ROLLING) {
    if (real_rows != rows_padded) return CP_ERR_INVALID_ARG;
    if (rows_padded > desc->capacity) return CP_ERR_CAPACITY;
  } else if ((int64_t)max_past + rows_padded > layout_limit(desc)) {
    return CP_ERR_CAPACITY;
  }
  const int64_t rows_total = (int64_t)desc->batch * rows_padded;
  if (rows_total > INT32_MAX || (int64_t)max_past + rows_padded > INT32_MAX) return CP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.hq = desc->num_q_heads;
  a.hkv = desc->num_kv_heads;
  a.d = desc->head_dim;
  a.group = a.hq / a.hkv;
  a.scale_log2 = scale_log2(desc);
  a.rows = SeqRows{desc->batch, rows_padded, nullptr};
  a.cache = make_cache(desc, block_table);
  a.past = seqlens_k;
  a.left_pad = desc->kind == CP_CACHE_ROLLING ? left_pad : nullptr;
  a.max_ctx = max_past + rows_padded;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.status = dev_status;
  r = run_attention(desc, a, rows_total, rows_padded, k_cache, v_cache, desc->batch, workspace, workspace_bytes, st);
  if (r != CP_OK) return r;
  if (commit) return launch_result(launch_commit(seqlens_k, a.rows, real_rows, nullptr, st));
  return CP_OK;
}

int cp_prefill_chunk(const cp_layer_desc* desc, const void* q, void* k_new, void* v_new, void* k_cache,
                     void* v_cache, int32_t* seqlens_k, const int32_t* block_table, const int32_t* left_pad,
                     int32_t rows_padded, int32_t real_rows, int32_t max_past, void* out, void* workspace,
                     size_t workspace_bytes, int32_t* dev_status, void* stream) {
  int r = check_desc(desc, true);
  if (r != CP_OK) return r;
  if (rows_padded <= 0 || real_rows <= 0 || real_rows > rows_padded || max_past < 0) return CP_ERR_INVALID_ARG;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !seqlens_k || !out) return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_PAGED && !block_table) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(out))
    return CP_ERR_INVALID_ARG;
  if (desc->kind == CP_CACHE_ROLLING) {
    if (real_rows != rows_padded) return CP_ERR_INVALID_ARG;
    if (rows_padded > desc->capacity) return CP_ERR_CAPACITY;
  } else if ((int64_t)max_past + rows_padded > layout_limit(desc)) {
    return CP_ERR_CAPACITY;
  }
  const int64_t rows_total = (int64_t)desc->batch * rows_padded;
  if (rows_total > INT32_MAX || (int64_t)max_past + rows_padded > INT32_MAX) return CP_ERR_UNSUPPORTED;
  // The copy of the lengths always; the split-KV partials only when the rows
  // take the split-KV path -- one row, or a short chunk of at most 16 / G rows
  // (checked here, before anything is enqueued).
  const int G0 = desc->num_q_heads / desc->num_kv_heads;
  if (desc->dtype != CP_F32 && !attn_tc_supported(desc->head_dim, G0, desc->dtype)) return CP_ERR_UNSUPPORTED;
  const bool decode_rows = rows_padded <= decode_max_rows(G0) && desc->dtype != CP_F32 &&
                           desc->kind != CP_CACHE_ROLLING && decode_supported(desc->head_dim, G0, desc->dtype);
  const int64_t snap = snapshot_bytes(desc->batch);
  const int64_t need =
      kControlBytes + snap +
      (decode_rows ? decode_ws_bytes(desc, max_past + rows_padded, (int64_t)desc->batch * rows_padded) : 0);
  if (workspace == nullptr || (int64_t)workspace_bytes < need || !aligned16(workspace)) return CP_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.hq = desc->num_q_heads;
  a.hkv = desc->num_kv_heads;
  a.d = desc->head_dim;
  a.group = a.hq / a.hkv;
  a.scale_log2 = scale_log2(desc);
  a.rows = SeqRows{desc->batch, rows_padded, nullptr};
  a.cache = make_cache(desc, block_table);
  a.left_pad = desc->kind == CP_CACHE_ROLLING ? left_pad : nullptr;
  a.max_ctx = max_past + rows_padded;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.status = dev_status;
  if (use_fused(desc, rows_padded)) {
    a.past = seqlens_k;  // read before any CTA takes its ticket
    a.ticket = static_cast<unsigned*>(workspace);
    a.commit_lens = seqlens_k;
    a.commit_add = real_rows;
    return run_fused(desc, a, rows_total, k_new, v_new, st);
  }
  if (desc->dtype == CP_F32 && desc->kind == CP_CACHE_CONTIG) {
    // fp32, contiguous: the fp32 kernel appends, attends and advances in one launch.
    a.past = seqlens_k;
    a.ticket = static_cast<unsigned*>(workspace);
    a.commit_lens = seqlens_k;
    a.commit_add = real_rows;
    a.min_rows = 1;
    a.fused = 1;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    return launch_result(launch_attn_f32(a, rows_padded, st));
  }
  int* past = reinterpret_cast<int*>(static_cast<char*>(workspace) + kControlBytes);

  AppendArgs ap;
  ap.hkv = desc->num_kv_heads;
  ap.d = desc->head_dim;
  ap.esize = esize_of(desc->dtype);
  ap.rows = SeqRows{desc->batch, rows_padded, nullptr};
  ap.cache = make_cache(desc, block_table);
  ap.past = seqlens_k;
  ap.max_ctx = max_past + rows_padded;
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_cache = k_cache;
  ap.v_cache = v_cache;
  ap.status = dev_status;
  ap.past_snapshot = past;
  r = launch_result(launch_kv_append(ap, (int)rows_total, st));
  if (r != CP_OK) return r;

  a.past = past;  // the snapshot: seqlens_k itself may then be advanced by the attention kernel
  // One launch for the attention and the commit when a single kernel takes
  // every row: the tensor-core kernel, or the fp32 one.
  const int G = desc->num_q_heads / desc->num_kv_heads;
  const bool tc_only = (desc->dtype == CP_F32 ||
                        (rows_padded > 1 && !decode_rows && attn_tc_supported(desc->head_dim, G, desc->dtype)));
  // Every row on one path (the tensor-core kernel, the fp32 one, or the
  // split-KV kernels of a short chunk): that path's kernel advances the lengths.
  const bool one_path = tc_only || decode_rows;
  if (one_path) {
    a.commit_lens = seqlens_k;
    a.commit_add = real_rows;
  }
  r = run_attention(desc, a, rows_total, rows_padded, k_cache, v_cache, desc->batch,
                    static_cast<char*>(workspace) + kControlBytes + snap,
                    (size_t)(workspace_bytes - kControlBytes - snap), st,
                    desc->kind == CP_CACHE_PAGED ? k_new : nullptr, desc->kind == CP_CACHE_PAGED ? v_new : nullptr);
  if (r != CP_OK) return r;
  if (!one_path) return launch_result(launch_commit(seqlens_k, a.rows, real_rows, nullptr, st));
  return CP_OK;
}

int cp_mixed_step(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new, void* k_pages,
                  void* v_pages, const int32_t* block_table, const int32_t* cu_rows, int32_t* past_len,
                  int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out, void* workspace,
                  size_t workspace_bytes, int32_t* dev_status, void* stream) {
  size_t need = 0;
  int r = cp::mixed_step_check(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len, num_seqs,
                               total_rows, max_ctx, out, &need);
  if (r != CP_OK) return r;
  if (total_rows == 0) return CP_OK;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))) return CP_ERR_WORKSPACE;
  return ragged_step(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len, num_seqs, total_rows,
                     max_ctx, out, workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int cp_mixed_step_overlap(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new,
                          void* k_pages, void* v_pages, const int32_t* block_table, const int32_t* cu_rows,
                          int32_t* past_len, int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream,
                          void* side_stream, void* fork_event, void* join_event) {
  size_t need = 0;
  int r = cp::mixed_step_check(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len, num_seqs,
                               total_rows, max_ctx, out, &need);
  if (r != CP_OK) return r;
  if (!side_stream || !fork_event || !join_event || side_stream == stream) return CP_ERR_INVALID_ARG;
  if (total_rows == 0) return CP_OK;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))) return CP_ERR_WORKSPACE;
  const ForkJoin fj{static_cast<cudaStream_t>(side_stream), static_cast<cudaEvent_t>(fork_event),
                    static_cast<cudaEvent_t>(join_event)};
  return ragged_step(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len, num_seqs, total_rows,
                     max_ctx, out, workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), &fj);
}

}  // extern "C"

namespace cp {
// The checks of cp_prefill_varlen (and its overlap form), in order; *need
// receives the workspace bytes the call needs.
int varlen_check(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new, void* k_cache,
                 void* v_cache, const int32_t* cu_rows, int32_t* seqlens_k, int32_t num_seqs, int32_t total_rows,
                 int32_t max_ctx, void* out, int64_t* need) {
  *need = 0;
  int r = check_desc(desc, true);
  if (r != CP_OK) return r;
  if (desc->kind != CP_CACHE_CONTIG) return CP_ERR_UNSUPPORTED;
  if (num_seqs <= 0 || num_seqs > desc->batch || total_rows < 0 || max_ctx <= 0) return CP_ERR_INVALID_ARG;
  if (total_rows == 0) return CP_OK;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !cu_rows || !seqlens_k || !out) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(out))
    return CP_ERR_INVALID_ARG;
  if ((int64_t)max_ctx > layout_limit(desc)) return CP_ERR_CAPACITY;
  const int G0 = desc->num_q_heads / desc->num_kv_heads;
  if (desc->dtype != CP_F32) {
    if (!attn_tc_supported(desc->head_dim, G0, desc->dtype)) return CP_ERR_UNSUPPORTED;
    if (decode_supported(desc->head_dim, G0, desc->dtype)) *need = decode_ws_bytes(desc, max_ctx, num_seqs);
  }
  return CP_OK;
}
}  // namespace cp

extern "C" {

int cp_prefill_varlen(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, const int32_t* cu_rows, int32_t* seqlens_k, int32_t num_seqs,
                      int32_t total_rows, int32_t max_ctx, void* out, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream) {
  int64_t need = 0;
  const int r = cp::varlen_check(desc, q, k_new, v_new, k_cache, v_cache, cu_rows, seqlens_k, num_seqs, total_rows,
                                 max_ctx, out, &need);
  if (r != CP_OK || total_rows == 0) return r;
  if (need > 0 && (workspace == nullptr || (int64_t)workspace_bytes < need || !aligned16(workspace)))
    return CP_ERR_WORKSPACE;
  return ragged_step(desc, q, k_new, v_new, k_cache, v_cache, nullptr, cu_rows, seqlens_k, num_seqs, total_rows,
                     max_ctx, out, workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int cp_prefill_varlen_overlap(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new,
                              void* k_cache, void* v_cache, const int32_t* cu_rows, int32_t* seqlens_k,
                              int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream, void* side_stream,
                              void* fork_event, void* join_event) {
  int64_t need = 0;
  const int r = cp::varlen_check(desc, q, k_new, v_new, k_cache, v_cache, cu_rows, seqlens_k, num_seqs, total_rows,
                                 max_ctx, out, &need);
  if (r != CP_OK) return r;
  if (!side_stream || !fork_event || !join_event || side_stream == stream) return CP_ERR_INVALID_ARG;
  if (total_rows == 0) return CP_OK;
  if (need > 0 && (workspace == nullptr || (int64_t)workspace_bytes < need || !aligned16(workspace)))
    return CP_ERR_WORKSPACE;
  const ForkJoin fj{static_cast<cudaStream_t>(side_stream), static_cast<cudaEvent_t>(fork_event),
                    static_cast<cudaEvent_t>(join_event)};
  return ragged_step(desc, q, k_new, v_new, k_cache, v_cache, nullptr, cu_rows, seqlens_k, num_seqs, total_rows,
                     max_ctx, out, workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), &fj);
}

}  // extern "C"
