/*
 * cp_api.h -- C ABI of the GB300 chunked-prefill causal attention library
 * (libcp.so, built for sm_103a).
 *
 * Sources cited below:
 *   [Wiki]     ONNX GenAI Wiki, "Chunked Prefill".
 *   [Horizon]  Horizon developer blog, "【大模型】Chunk Prefill——把一次算不动的事拆成多次".
 *   [Glossary] Ultralytics glossary, "Chunked Prefill".
 *
 * Conventions shared by every entry point:
 *   - Pointers named as device pointers must point to GPU memory of the
 *     current device; the caller allocates and owns every buffer.  The
 *     library allocates nothing and keeps no state between calls, so calls on
 *     different streams are independent.  "host" pointers are read before the
 *     call returns.
 *   - Layouts are dense row-major with the last dimension contiguous:
 *       q, out           [B, R, Hq, D]   (cp_prefill_chunk_attn)
 *                        [T, Hq, D]      (cp_mixed_step, cp_prefill_varlen)
 *       k_new, v_new     [B, R, Hkv, D]  (cp_kv_append), [T, Hkv, D] (mixed)
 *       contiguous cache [B, Hkv, capacity, D]
 *       rolling cache    [B, Hkv, capacity, D]
 *       paged pool       [num_pages, Hkv, page_size, D]
 *       block_table      int32 [B or S, max_blocks], page ids of each sequence
 *     Element type is cp_layer_desc.dtype for all of q, k, v, caches and out.
 *     Device pointers must be 16-byte aligned.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL =
 *     the legacy default stream).
 *   - Errors: every argument is checked on the host before anything is
 *     enqueued; on a bad argument the call returns a negative cp_status and
 *     launches nothing.  CP_ERR_CUDA is returned if a launch reports an error.
 *     Values that live on the device (seqlens_k, past_len, block table
 *     entries) are checked by the kernels against the host bounds given in
 *     the call: an out-of-range value is never dereferenced -- the affected
 *     rows are skipped and, if `dev_status` is not NULL, a CP_DEV_* bit is
 *     OR-ed into *dev_status (an int32 in device memory the caller zeroes and
 *     reads back after synchronizing).  No kernel asserts or traps; every
 *     wait inside a kernel is bounded and reports CP_DEV_TIMEOUT.
 */
#ifndef CP_API_H
#define CP_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CP_ABI_VERSION 1

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1, /* malformed argument (null, negative, misaligned, ...) */
  CP_ERR_UNSUPPORTED = -2, /* well-formed but outside what the kernels implement  */
  CP_ERR_CAPACITY = -3,    /* rows would not fit in the cache / pages / table      */
  CP_ERR_CUDA = -4,        /* a CUDA launch or query failed                         */
  CP_ERR_WORKSPACE = -5    /* workspace missing or smaller than cp_workspace_size   */
} cp_status;

/* Bits OR-ed into *dev_status by kernels. */
#define CP_DEV_BOUNDS 1  /* a device-side length or page id was out of range   */
#define CP_DEV_TIMEOUT 2 /* a bounded wait inside a kernel gave up             */

typedef enum { CP_F32 = 0, CP_BF16 = 1, CP_F16 = 2 } cp_dtype;

/* Cache layouts.
 * CONTIG : fixed physical capacity, slot = absolute position ([Wiki] 一.3: the
 *          past K/V stay bound at physical capacity; the valid length travels
 *          separately in seqlens_k).
 * ROLLING: right-aligned window of the newest `capacity` positions ([Horizon]
 *          2-4).  Position a lives in slot a mod capacity, so the window's
 *          rotation is implied by seqlens_k and needs no separate state.
 * PAGED  : fixed-size pages listed in a block table ([Glossary] "Related
 *          techniques", PagedAttention). */
typedef enum { CP_CACHE_CONTIG = 0, CP_CACHE_ROLLING = 1, CP_CACHE_PAGED = 2 } cp_cache_kind;

typedef struct {
  int32_t dtype;        /* cp_dtype                                            */
  int32_t batch;        /* B, sequences in a cp_kv_append / prefill call        */
  int32_t num_q_heads;  /* Hq                                                   */
  int32_t num_kv_heads; /* Hkv; Hq % Hkv == 0 (GroupQueryAttention, [Wiki] 一.3) */
  int32_t head_dim;     /* D: 64 or 128                                         */
  int32_t kind;         /* cp_cache_kind                                        */
  int32_t capacity;     /* CONTIG/ROLLING: slots per (sequence, KV head)        */
  int32_t page_size;    /* PAGED: tokens per page (16, 32, 64 or 128)           */
  int32_t num_pages;    /* PAGED: pages in the pool                             */
  int32_t max_blocks;   /* PAGED: columns of block_table                        */
  float scale;          /* softmax scale; 0 selects 1/sqrt(head_dim)            */
} cp_layer_desc;

/* cp_kv_append -- write a chunk's new K/V rows into the cache.
 *
 * [Wiki] 一.1: chunk k writes its own positions and never revisits or
 * rewrites an earlier slot.  [Horizon] 3: in rolling mode the new rows replace
 * the oldest ones.  [Glossary]: in paged mode a sequence's cache grows page by
 * page.
 *   k_new, v_new  device [B, rows, Hkv, D]
 *   rows          rows per sequence (the padded width R when padding is used)
 *   k_cache, v_cache  device cache of desc->kind (layouts above)
 *   seqlens_k     device int32 [B]: valid length = absolute position of row 0.
 *                 Not modified (cp_prefill_chunk_attn commits it).
 *   block_table   device int32 [B, max_blocks] (PAGED only, else NULL)
 *   max_past      host bound on every seqlens_k[b]; CONTIG needs
 *                 max_past + rows <= capacity, ROLLING needs rows <= capacity,
 *                 PAGED needs max_past + rows <= max_blocks * page_size.
 * Row t of sequence b goes to absolute position seqlens_k[b] + t:
 * CONTIG slot = position; ROLLING slot = position mod capacity; PAGED page =
 * block_table[b][position / page_size], offset position % page_size.
 * Bit-exact copy; nothing else in the cache is touched. */
int cp_kv_append(const cp_layer_desc* desc, const void* k_new, const void* v_new,
                 int32_t rows, void* k_cache, void* v_cache, const int32_t* seqlens_k,
                 const int32_t* block_table, int32_t max_past, int32_t* dev_status,
                 void* stream);

/* cp_pad_chunk -- widen a chunk in place to its query-width tier.
 *
 * [Wiki] 四: the rows of a forward are rounded up to a ladder tier and the
 * extra rows repeat the last real token; every per-token input of shape
 * [1, rows, ...] is widened the same way.  For each sequence b, rows
 * [real_rows, rows_padded) of q [B, rows_padded, Hq, D] and of k_new, v_new
 * [B, rows_padded, Hkv, D] (device) are overwritten with copies of row
 * real_rows - 1; rows below real_rows are not touched.  Any of the three
 * pointers may be NULL to skip that tensor.  Bit-exact copy. */
int cp_pad_chunk(const cp_layer_desc* desc, void* q, void* k_new, void* v_new, int32_t real_rows,
                 int32_t rows_padded, void* stream);

/* cp_prefill_chunk_attn -- causal attention of one chunk of query rows.
 *
 * Row i of sequence b is the query at absolute position p = seqlens_k[b] + i
 * and attends to every cached key before the chunk plus its own causal
 * triangle: keys at positions [0, p] ([Wiki] 一.2; [Glossary] "How chunked
 * prefill works": the chunk mask is the lower triangle shifted by the chunk
 * start).  The chunk's K/V must already be in the cache (cp_kv_append).
 *   O[b,i,h] = sum_j softmax_j(scale * q[b,i,h] . k_j) v_j over visible j,
 *   KV head of query head h = h / (Hq / Hkv).
 * ROLLING ([Horizon] 3-4): the cache holds the newest `capacity` positions;
 * key position a is visible iff a >= left_pad[b], a >= 0, a is still in the
 * window and a <= p.  (The page adds -32768 to masked scores; for a row with
 * at least one visible key that weight underflows to exactly 0, so excluding
 * the slot gives the same result.  A row with no visible key -- a left-pad
 * query -- gets output 0.)
 * Paths: bf16/fp16 chunks of at most 16 / G rows per sequence (a decode row,
 * or k draft tokens verified in one pass) take the memory-bound split-KV
 * path, every row of a sequence sharing one read of its K/V (not ROLLING);
 * longer chunks take the tensor-core path; fp32 a SIMT path.
 *   q, out        device [B, rows_padded, Hq, D]; pad rows' outputs are
 *                 written but unspecified ([Wiki] 四: results are cut back to
 *                 the real rows)
 *   seqlens_k     device int32 [B]; if commit != 0 it is advanced by real_rows
 *                 after the attention ([Wiki] 四: rewind to past + real rows;
 *                 the pad rows' K/V stay beyond it until the next chunk
 *                 overwrites them)
 *   left_pad      device int32 [B] (ROLLING, may be NULL = 0), else NULL
 *   rows_padded   R, rows per sequence in q/out (query-width ladder tier)
 *   real_rows     r <= R; ROLLING requires r == R (a pad row would evict a
 *                 live slot)
 *   max_past      host bound on seqlens_k[b] (same rule as cp_kv_append)
 *   workspace     device scratch of at least
 *                 cp_workspace_size(desc, B * R, max_past + R, B) bytes
 *                 (may be NULL when that size is 0) */
int cp_prefill_chunk_attn(const cp_layer_desc* desc, const void* q, const void* k_cache,
                          const void* v_cache, int32_t* seqlens_k, const int32_t* block_table,
                          const int32_t* left_pad, int32_t rows_padded, int32_t real_rows,
                          int32_t max_past, void* out, void* workspace, size_t workspace_bytes,
                          int32_t commit, int32_t* dev_status, void* stream);

/* cp_prefill_chunk -- one chunk of a prompt in one call: cp_kv_append of the
 * chunk's K/V rows, cp_prefill_chunk_attn of its query rows, and the advance of
 * seqlens_k by real_rows, with the same arguments and results as those two
 * calls made back to back with commit = 1 ([Glossary] "How chunked prefill
 * works": each chunk's K/V join the cache and its rows attend to the cache).
 * For a contiguous cache in bf16/fp16 with more rows per sequence than the
 * split-KV path takes (16 / G), for a contiguous cache in fp32, and for a
 * rolling cache in bf16/fp16 wider than 128 slots with rows <= capacity - 128,
 * this is one kernel launch: the kernel reads the chunk's own keys straight
 * from k_new / v_new, copies those rows into the cache (ring: slot position
 * mod capacity), and the last of its CTAs to have read seqlens_k advances it.
 * Other cases take an append launch followed by the attention.
 *   q, out        device [B, rows_padded, Hq, D]
 *   k_new, v_new  device [B, rows_padded, Hkv, D] (rows [real_rows,
 *                 rows_padded) are appended too: cp_pad_chunk fills them); they
 *                 must not alias the cache or out
 *   workspace     device scratch, 16-byte aligned, of at least
 *                 cp_workspace_size(desc, B * R, max_past + R, B) bytes (that
 *                 size always suffices).  Its first 256 bytes are a control
 *                 block that must be zero before the first call that uses this
 *                 workspace (allocate it zeroed); every call leaves it zero.
 *                 Calls whose work overlaps on the GPU need separate workspaces.
 * Other arguments as in cp_prefill_chunk_attn. */
int cp_prefill_chunk(const cp_layer_desc* desc, const void* q, void* k_new, void* v_new, void* k_cache,
                     void* v_cache, int32_t* seqlens_k, const int32_t* block_table,
                     const int32_t* left_pad, int32_t rows_padded, int32_t real_rows, int32_t max_past,
                     void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream);

/* cp_mixed_step -- one token-budget step over a paged cache.
 *
 * [Glossary] "How chunked prefill works": a step holds one row for every
 * running decode plus chunks of waiting prompts; mixing them uses the compute
 * that decode rows leave idle.  The call appends every row's K/V into its
 * sequence's pages, then computes causal attention for every row (decode rows
 * -- sequences with one row -- on a memory-bound split-KV path, prompt chunks on
 * the tensor-core path), then advances past_len[s] by the sequence's rows.
 *   desc->kind must be CP_CACHE_PAGED; desc->batch is ignored.
 *   q, out        device [T, Hq, D];  k_new, v_new device [T, Hkv, D]
 *   k_pages, v_pages  device pools [num_pages, Hkv, page_size, D]
 *   block_table   device int32 [num_seqs, max_blocks]
 *   cu_rows       device int32 [num_seqs + 1]: rows of sequence s are
 *                 [cu_rows[s], cu_rows[s+1]); cu_rows[num_seqs] == T.  Every
 *                 listed sequence has at least one row (a sequence with no
 *                 rows in this step is left out of the call); the host relies
 *                 on it to bound rows per sequence by T - num_seqs + 1, and a
 *                 sequence with no rows sets CP_DEV_BOUNDS in *dev_status
 *   past_len      device int32 [num_seqs]: positions already cached
 *   max_ctx       host bound on past_len[s] + rows of s (<= max_blocks*page_size)
 *   workspace     device scratch, 16-byte aligned, of at least
 *                 cp_workspace_size(desc, T, max_ctx, num_seqs) bytes (that size
 *                 always suffices; fp32 layers need none and may pass NULL) */
int cp_mixed_step(const cp_layer_desc* desc, const void* q, const void* k_new,
                  const void* v_new, void* k_pages, void* v_pages, const int32_t* block_table,
                  const int32_t* cu_rows, int32_t* past_len, int32_t num_seqs,
                  int32_t total_rows, int32_t max_ctx, void* out, void* workspace,
                  size_t workspace_bytes, int32_t* dev_status, void* stream);

/* cp_mixed_step_overlap -- cp_mixed_step with its two attention paths running
 * side by side.
 *
 * [Glossary] "How chunked prefill works": the decode rows of a mixed step are
 * memory-bound and the prompt chunks compute-bound, so the GPU can serve both
 * at once.  This call does what cp_mixed_step does, with the same arguments,
 * checks, status codes and results (bit for bit), but when a step has both
 * decode rows and prompt chunks it launches the split-KV kernels on
 * `side_stream` and the tensor-core kernel on `stream` in between:
 *   stream:      append -> record(fork_event) -> tensor-core attention
 *                -> wait(join_event) -> length advance
 *   side_stream: wait(fork_event) -> split-KV + combine -> record(join_event)
 * A step with only one kind of row runs everything on `stream`.  On this GPU a
 * tensor-core CTA takes its SM's whole register file, so the two kinds of kernel
 * share the GPU only where one grid drains and the other fills: the step may
 * come out a little shorter or a little longer than with cp_mixed_step.
 *   side_stream   a CUDA stream of the same device, not `stream` (caller-owned;
 *                 work the caller queued there before the call runs first)
 *   fork_event, join_event  caller-owned cudaEvent_t handles (created with
 *                 cudaEventDisableTiming is best); the call records them, so
 *                 they must not be waited on by other work until it returns.
 * Under stream capture both streams join back into `stream` before the call
 * returns, so the step captures as one graph.  NULL side_stream or events, or
 * side_stream == stream, return CP_ERR_INVALID_ARG. */
int cp_mixed_step_overlap(const cp_layer_desc* desc, const void* q, const void* k_new,
                          const void* v_new, void* k_pages, void* v_pages,
                          const int32_t* block_table, const int32_t* cu_rows, int32_t* past_len,
                          int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          void* stream, void* side_stream, void* fork_event, void* join_event);

/* cp_prefill_varlen -- one step of several prompts with ragged rows over a
 * contiguous cache.
 *
 * [Glossary] "How chunked prefill works": a step is filled with chunks of
 * several waiting prompts (and one row per running decode), each sequence
 * with its own row count and its own cached length.  This is cp_mixed_step
 * for a cache at fixed physical capacity ([Wiki] 一.3): every row's K/V is
 * appended at slots seqlens_k[s] .. seqlens_k[s] + rows(s) - 1 of sequence s,
 * then row i of s attends causally to slots [0, seqlens_k[s] + i] (one-row
 * sequences on the split-KV decode path, the others on the tensor-core
 * path), then seqlens_k[s] advances by rows(s).  No query padding: every row
 * is real.
 *   desc->kind must be CP_CACHE_CONTIG; sequences 0 .. num_seqs-1 of the
 *                 cache take part (num_seqs <= desc->batch).
 *   q, out        device [T, Hq, D];  k_new, v_new device [T, Hkv, D]
 *   k_cache, v_cache  device [desc->batch, Hkv, capacity, D]
 *   cu_rows       device int32 [num_seqs + 1] as in cp_mixed_step (every
 *                 listed sequence has at least one row)
 *   seqlens_k     device int32 [num_seqs]: valid slots of each sequence
 *   max_ctx       host bound on seqlens_k[s] + rows(s) (<= capacity; a
 *                 larger device value sets CP_DEV_BOUNDS and its rows are
 *                 skipped)
 *   workspace     device scratch, 16-byte aligned, of at least
 *                 cp_workspace_size(desc, T, max_ctx, num_seqs) bytes (fp32
 *                 layers need none) */
int cp_prefill_varlen(const cp_layer_desc* desc, const void* q, const void* k_new,
                      const void* v_new, void* k_cache, void* v_cache, const int32_t* cu_rows,
                      int32_t* seqlens_k, int32_t num_seqs, int32_t total_rows, int32_t max_ctx,
                      void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream);

/* cp_prefill_varlen_overlap -- cp_prefill_varlen with its one-row sequences
 * on a side stream.
 *
 * The same call as cp_prefill_varlen (same arguments, checks, status codes
 * and results, bit for bit), but when a step has both one-row sequences
 * (split-KV path) and longer ones (tensor-core path), the split-KV kernels run
 * on `side_stream` beside the tensor-core kernel, forked after the append and
 * joined before the length advance, exactly as cp_mixed_step_overlap does.
 * side_stream, fork_event and join_event as in cp_mixed_step_overlap (NULL,
 * or side_stream == stream, returns CP_ERR_INVALID_ARG). */
int cp_prefill_varlen_overlap(const cp_layer_desc* desc, const void* q, const void* k_new,
                              const void* v_new, void* k_cache, void* v_cache, const int32_t* cu_rows,
                              int32_t* seqlens_k, int32_t num_seqs, int32_t total_rows, int32_t max_ctx,
                              void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream, void* side_stream, void* fork_event, void* join_event);

/* cp_mixed_step_noalloc -- cp_mixed_step for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it is a convenience of
 * this library's interface.  Some callers cannot allocate device memory or hand
 * the library a workspace: serving engines that reserve all device memory up
 * front and forbid allocation on the request path, plugins that receive only
 * input and output tensors from a host framework that owns every allocation,
 * and code running where cudaMalloc is not allowed (for example inside a
 * stream callback).  This is cp_mixed_step with its split-KV scratch taken from
 * a fixed array of cp_noalloc_scratch_bytes() bytes (8 MiB) compiled into the
 * library.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *   Arguments, checks, status codes and results are those of cp_mixed_step,
 *   without the workspace.  A step whose split-KV partials (the workspace
 *   cp_mixed_step would use for it) exceed the array is refused with
 *   CP_ERR_WORKSPACE before anything is enqueued.
 *   Set-up: the array lives in its own CUDA module.  With the CUDA runtime's
 *   lazy module loading (the default) that module -- and so the array's 8 MiB
 *   of device memory -- is loaded on a device by this entry point's first call
 *   there, which also looks up the array's device address (once per device,
 *   with that device current).  Make that first call on each device during
 *   set-up (a small warm-up step), before reserving the rest of the device's
 *   memory and before any stream capture.  Calls after cudaDeviceReset are not
 *   supported (the looked-up address belongs to the reset context).
 *   Every call uses the same array, which keeps the last call's contents:
 *   each call writes every entry it uses before reading it.
 *   Calls whose work overlaps on the GPU -- on different streams or from
 *   different host threads -- race on the array; the caller must serialise
 *   them. */
int cp_mixed_step_noalloc(const cp_layer_desc* desc, const void* q, const void* k_new,
                          const void* v_new, void* k_pages, void* v_pages,
                          const int32_t* block_table, const int32_t* cu_rows, int32_t* past_len,
                          int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out,
                          int32_t* dev_status, void* stream);

/* cp_noalloc_scratch_bytes -- size of the fixed scratch array used by
 * cp_mixed_step_noalloc (no GPU work). */
size_t cp_noalloc_scratch_bytes(void);

/* cp_workspace_size -- bytes of device scratch the attention calls need for up
 * to `max_rows` query rows, contexts of up to `max_ctx` keys and `num_seqs`
 * sequences: a 256-byte control block and a copy of the sequences' lengths
 * (cp_prefill_chunk; the control block must be zero before first use, see
 * there) and the split-KV partial results: for each sequence, one row's, or
 * up to 16 / G rows' when a call's rows per sequence are that few (short
 * chunks, e.g. k draft tokens verified in one pass, take the split-KV path
 * together); for 16-bit layers, also room for the work list of a ragged call
 * (cp_mixed_step, cp_mixed_step_overlap, cp_prefill_varlen): 8 bytes per pair
 * of 2 * 128 / G query tokens plus 8 per sequence.  A ragged call keeps the
 * list after its split-KV partials and uses it only when the workspace has
 * room: it then hands the tensor-core kernel's clusters the pairs that see
 * the most keys first (results are the same bit for bit either way). */
size_t cp_workspace_size(const cp_layer_desc* desc, int32_t max_rows, int32_t max_ctx,
                         int32_t num_seqs);

/* ---- host-side integer helpers (no GPU work) ---- */

/* cp_chunk_plan -- chunk sizes of an n_tokens prompt at width `chunk`
 * ([Wiki] 三: every chunk is `chunk` wide except the last, which takes the
 * remainder).  Writes up to `cap` sizes to host `sizes` and returns the
 * number of chunks (which may exceed cap), or a negative cp_status. */
int32_t cp_chunk_plan(int32_t n_tokens, int32_t chunk, int32_t* sizes, int32_t cap);

/* cp_query_ladder -- the query-width tiers of chunk width `chunk` ([Wiki] 四
 * and 六: three evenly spaced tiers whose step ceil(chunk/3) is rounded up
 * so the top tier is exactly `chunk`; {171,342,512} for 512).  Writes the
 * distinct tiers (1 to 3) to host `tiers[3]` and returns their count. */
int32_t cp_query_ladder(int32_t chunk, int32_t* tiers);

/* cp_query_width -- smallest tier >= real_rows (1 <= real_rows <= chunk), or a
 * negative cp_status. */
int32_t cp_query_width(int32_t real_rows, int32_t chunk);

/* cp_aligned_length -- n_real rounded up to a multiple of the chunk size c
 * ([Horizon] 5: the prompt is left-padded to a multiple of chunk_size). */
int32_t cp_aligned_length(int32_t n_real, int32_t c);

/* cp_rolling_mask -- materialise the per-chunk additive mask [c, C] of
 * [Horizon] 4 into host `out` (row-major floats): row i is the query at
 * absolute position chunk_idx*c + i, slot j holds position
 * (chunk_idx+1)*c - C + j; the entry is 0 when that position exists, is not
 * a left-pad position and is not in the future, else -32768.  The kernels
 * never materialise it; it is here for tests and callers that want the
 * tensor.  Returns CP_OK or a negative cp_status. */
int cp_rolling_mask(int32_t c, int32_t C, int32_t chunk_idx, int32_t left_pad, float* out);

/* One entry of a token-budget plan.  Decode rows have start == -1, rows == 1. */
typedef struct {
  int32_t step;  /* step index, from 0                                     */
  int32_t seq;   /* running decodes 0..n_running-1, prompt i = n_running+i */
  int32_t start; /* first prompt token of the chunk, -1 for a decode row   */
  int32_t rows;  /* rows of this entry in the step                         */
} cp_sched_entry;

/* cp_schedule -- token-budget step plan ([Glossary] "How chunked prefill
 * works"): each step gives one row to every running decode first, then fills
 * the remaining budget with chunks of the waiting prompts in arrival order; a
 * prompt that does not fit continues next step and decodes from the step
 * after its last chunk.  Entries of a step are ordered decodes first (by seq
 * id), then prompt chunks.  Writes up to `cap` entries to host `out` and
 * returns the total entry count (may exceed cap), or a negative cp_status
 * (CP_ERR_INVALID_ARG if the budget leaves no room for prompt tokens). */
int32_t cp_schedule(int32_t budget, int32_t n_running, const int32_t* prompt_lens,
                    int32_t n_prompts, cp_sched_entry* out, int32_t cap);

/* cp_status_string -- static text for a cp_status value. */
const char* cp_status_string(int32_t status);

/* cp_selftest_bounded_wait -- checks, on the device, the bounded wait that
 * every kernel of this library uses for its barriers (no page defines it:
 * it is this library's failure-detection path).  One warp waits on a
 * barrier that nothing completes; the wait gives up after the library's wait
 * limit (4 s), ORs CP_DEV_TIMEOUT into *dev_status and raises the CTA's abort
 * flag, and a second wait returns at once.  No fault, no trap: the context
 * stays usable.  Asynchronous on `stream`; takes the wait limit to finish.
 *   dev_status  device int32, OR-ed with CP_DEV_TIMEOUT
 *   dev_out     device uint64[5], 8-byte aligned: first wait succeeded (0/1),
 *               its duration in ns, second wait succeeded (0/1), its
 *               duration in ns, the abort flag at the end (0/1)
 * Returns CP_ERR_INVALID_ARG for a null or misaligned pointer, CP_ERR_CUDA if
 * the launch fails, else CP_OK. */
int cp_selftest_bounded_wait(int32_t* dev_status, uint64_t* dev_out, void* stream);

/* cp_abi_version -- CP_ABI_VERSION of the built library. */
int32_t cp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CP_API_H */
