// attn_tc.cu -- chunk attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ([Wiki] 一.2; [Glossary] "How chunked prefill works"): row i
// of a chunk is the query at absolute position p = past + i and attends to
// the keys at positions [0, p] -- the cached prefix plus its own causal
// triangle -- over a cache at fixed physical capacity, a paged pool, or a
// right-aligned rolling window ([Horizon] 3-4).
//
// Work decomposition.  GroupQueryAttention packs the G = Hq/Hkv query heads of
// one KV head into 128-row Q tiles: 128/G consecutive tokens x G heads, row
// m <-> (token m / G, head m % G), so every K/V tile serves all heads of the
// group.  A cluster of two CTAs owns a pair of Q tiles (256 rows); both CTAs
// hold both Q tiles, and the KV tiles (128 keys, starting at absolute key 0)
// are split between them by parity: rank 0 takes tiles 0, 2, 4, ..., rank 1
// tiles 1, 3, 5, ....  Each CTA thus multiplies every K/V tile it loads into
// 256 query rows -- the shared-memory fill rate from L2 (about 30 bytes per
// clock per SM on this part) would otherwise cap the tensor pipe -- while a
// chunk still spreads over as many SMs as it has 128-row tiles.  Tile
// boundaries and the parity split depend only on absolute positions, so a
// padded and an unpadded run of the same rows do identical arithmetic; tiles
// past the pair's last query position are never loaded (causal tile skip).
// On a contiguous cache the tile that straddles `past` is walked twice, once
// for its cached keys and once for the chunk's own (see Walk), so that the
// fused append below and a separate append do the same arithmetic.
//
// Fused append (contiguous caches): the walks over the chunk's own keys read
// them straight from k_new / v_new, warp 2 copies the K/V rows of its Q tile's
// tokens into their cache slots ([Wiki] 一.1), and the last CTA to take a
// ticket advances seqlens_k by the real rows ([Wiki] 四) -- append, attention
// and commit in one launch.
//
// Warp roles (384 threads per CTA, three warpgroups):
//   warp 0      TMA producer: both Q tiles once, then this CTA's K and V tiles
//               in a 2-stage ring, one stage = one K tile + one V tile, each
//               with its own barrier (paged caches: one box per page and lane;
//               at head_dim 128 a box holds both 64-column halves of a page and
//               the stage takes the page layout, 8-row groups [half][8][128 B],
//               which the MMA descriptors of that instantiation follow).  The
//               first stage is issued as Q0, K, Q1, V, so the first MMA waits
//               for a quarter of the start-up bytes.
//   warp 1      TMEM allocator and MMA issuer (one elected lane).  Per KV tile:
//               S0 = Q0 K^T, S1 = Q1 K^T (A, B K-major in shared memory);
//               O0 += P0 V, O1 += P1 V (A = P in TMEM, B = V MN-major).
//   warp 2      fused append: copies this CTA's Q tile's K/V rows into the cache.
//   warp 3      takes the CTA's ticket (fused append); both fill the control
//               warpgroup, whose registers go to the softmax warpgroups.
//   warps 4-7   softmax group 0 (Q tile 0);  warps 8-11 softmax group 1 (Q tile 1).
// TMEM (512 columns): group w uses [256w, 256w+128) for S/P, [256w+128, +D) for O.
// Thread m of a group owns row m (TMEM lane m): it reads its S row, masks by
// absolute position, exponentiates in the log2 domain against a running max,
// writes P (16-bit) over the S columns, and rescales its O row only when its
// own max has grown by more than kRescaleLog2 (a row-local decision).
//
// Ordering: the MMA warp issues S_w(i+1) after O_w += P_w(i) V(i), and tcgen05
// operations from one thread complete in issue order, so when group w sees
// S_w(i+1) complete, its P V of tile i has completed too: O_w is then safe to
// rescale and P_w(i+1) may overwrite P_w(i).
//
// Merge: each CTA's partial (max, sum, unnormalised O) per row is combined in
// a fixed order (even-tile half first): rank r finishes the rows of Q tile r.
// Once a CTA's own MMAs are complete it tells its peer (a remote mbarrier
// arrive) that its K/V stages may receive; the peer's group for the other Q
// tile stages its partial O rows in its own K stages, 32 columns at a time
// (16-byte pieces XOR-swizzled by row, so the row-per-thread stores are
// conflict-free), and sends each 16 KB chunk with a bulk shared-to-shared
// copy as soon as it is staged, completed on one of the receiver's mbarriers.
// The receiver combines each chunk as it lands, writes the finished 16-bit
// rows into its Q buffer in the TMA layout and stores the tile with a TMA
// tensor store.
//
// Keys beyond the written length inside the last tile may hold stale or
// poisoned bytes; their scores are masked and the MMA warp zeroes those V rows
// before P V, so 0 * garbage never reaches O.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kThreads = 384;
// Register split: the kernel is compiled at kRegsLaunch per thread (the most
// 384 threads may have); the control warpgroup (warps 0-3) then drops to
// kRegsControl and hands the rest to the two softmax warpgroups.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax == kThreads * kRegsLaunch, "the split must add up");
constexpr int kStages = 2;
constexpr uint32_t kBlockBytes = 128 * 128;  // [128 rows][64 x 16-bit] = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;         // O is rescaled when the max grows by > 2^8

struct __align__(16) TcBarriers {
  uint64_t q_full[2];                                          // Q tile 0 / Q tile 1 landed
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];  // a stage holds one K tile and one V tile
  uint64_t s_full[2], p_ready[2];
  uint64_t o_final;
  uint64_t merge_full[4];  // column chunk c of the peer's partial for this CTA's rows has landed
  uint64_t peer_free;   // the peer's K/V stages may receive this CTA's partial
  uint32_t tmem_base;
  int abort;
  __align__(16) float peer_ml[256];  // the peer's partial max [0, 128) and sum [128, 256) for this CTA's rows
  __align__(16) float out_ml[256];   // this CTA's partial max / sum for the peer's rows (sent)
};

template <int D>
struct TcSmem {
  static constexpr int DB = D / 64;
  static constexpr uint32_t q_off = 0;                                   // 2 Q tiles
  static constexpr uint32_t k_off = q_off + 2 * DB * kBlockBytes;        // K stages
  static constexpr uint32_t v_off = k_off + kStages * DB * kBlockBytes;  // V stages
  static constexpr uint32_t bar_off = v_off + kStages * DB * kBlockBytes;
  static constexpr uint32_t bytes = bar_off + sizeof(TcBarriers);
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
  // After the main loop the K stages hold this CTA's outgoing partial O rows
  // and the V stages the peer's incoming ones: 128 rows x D fp32 each, as
  // D/32 column chunks of 16 KB that travel (and are combined) one by one.
  static constexpr uint32_t kMergeBytes = 128u * D * 4u;
  static constexpr int kMergeChunks = D / 32;
  static constexpr uint32_t kChunkBytes = 128u * 32u * 4u;
  static_assert(kStages * DB * kBlockBytes == kMergeBytes, "a merge buffer is exactly the K (or V) stages");
  static_assert(kMergeChunks <= 4, "merge_full has one barrier per column chunk");
};

// Byte offset of 16-byte piece e (columns 32c + 4e .. +3) of row m in a merge
// buffer: chunk c is a contiguous [128 rows][128 B] block, and the pieces of
// a row are XOR-swizzled by (m mod 8), so the 8 rows a quarter-warp touches at
// once fall on distinct banks.
__device__ __forceinline__ uint32_t merge_off(int m, int c, int e) {
  return (uint32_t)c * (128u * 128u) + (uint32_t)m * 128u + (uint32_t)((e ^ (m & 7)) * 16);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Which (sequence, first token) a cluster owns; a pair covers 2*rpt tokens.
// With a work list it is entry w; otherwise, within a sequence the pairs are
// handed out last-first, so the pairs with the most keys start earliest.  Every warp of the CTA calls this with all
// lanes: for ragged rows each warp scans the sequences 32 at a time (one
// coalesced round of loads per 32 sequences, a shuffle prefix sum of their
// pair counts), so the lookup costs a few memory latencies, not one per
// sequence.
__device__ __forceinline__ bool find_pair(const AttnArgs& a, int ppt, int w, int& s, int& t0) {
  if (a.pair_order) {
    const int2 e = a.pair_order[w];
    s = e.x;
    t0 = e.y;
    return e.x >= 0;
  }
  if (a.rows.rows_uniform > 0) {
    const int np = (a.rows.rows_uniform + ppt - 1) / ppt;
    const int pair = np - 1 - w / a.rows.num_seqs;
    s = w % a.rows.num_seqs;
    if (pair < 0) return false;
    t0 = pair * ppt;
    return true;
  }
  const int lane = threadIdx.x & 31;
  for (int q0 = 0; q0 < a.rows.num_seqs; q0 += 32) {
    const int q = q0 + lane;
    int np = 0;
    if (q < a.rows.num_seqs) {
      const int r = seq_rows(a.rows, q);
      np = r < a.min_rows ? 0 : (r + ppt - 1) / ppt;
    }
    int inc = np;  // inclusive prefix sum over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    if (w < tot) {
      const int L = __ffs(__ballot_sync(0xffffffffu, inc > w)) - 1;
      const int before = __shfl_sync(0xffffffffu, inc - np, L);
      const int npl = __shfl_sync(0xffffffffu, np, L);
      s = q0 + L;
      t0 = (npl - 1 - (w - before)) * ppt;
      return true;
    }
    w -= tot;
  }
  return false;
}

// The KV tiles a pair walks.  Tile t holds key indices [128t, 128t + 128).  On
// a contiguous cache the tiles below `past` hold cached keys and those at or
// above it the call's own rows; a tile that straddles `past` is walked twice
// (its cached keys, then its new ones), whether or not the append is fused, so
// the fused and the separate-call paths do the same arithmetic.  Other layouts
// walk each tile once.  Virtual tile j goes to CTA rank j % 2.
struct Walk {
  bool split;
  int past, n_valid, tp, count;
  bool straddle;
  __device__ __forceinline__ Walk(bool contig, int past_, int n_valid_, int ntiles) {
    split = contig;
    past = past_;
    n_valid = n_valid_;
    tp = past_ / kTcBlockN;
    straddle = contig && (past_ % kTcBlockN) != 0;
    count = ntiles + (straddle ? 1 : 0);
  }
  __device__ __forceinline__ void at(int j, int& tile, bool& is_new) const {
    if (!split || j < tp) {
      tile = j;
      is_new = false;
    } else if (straddle) {
      tile = j == tp ? tp : j - 1;
      is_new = j != tp;
    } else {
      tile = j;
      is_new = true;
    }
  }
  // Key indices [lo, hi) of the tile that belong to this walk.
  __device__ __forceinline__ void range(int tile, bool is_new, int& lo, int& hi) const {
    const int j0 = tile * kTcBlockN;
    if (!split) {
      lo = j0;
      hi = min(j0 + kTcBlockN, n_valid);
    } else {
      lo = is_new ? max(j0, past) : j0;
      hi = is_new ? min(j0 + kTcBlockN, n_valid) : min(j0 + kTcBlockN, past);
    }
  }
};

// The walks of a ring cache's physical slots [0, nkeys).  The call's rows are
// positions [past, past + rows), in slots (past + t) mod cap: one range of
// slots that wraps only at the ring's end.  When the ring is wider than a tile
// and rows <= cap - 128 (so no tile holds both ends of a wrapped range), a tile
// that holds cached and new slots is walked twice, its cached slots and then
// its new ones, whether or not the append is fused (so both paths do the same
// arithmetic), and every tile's new slots form one contiguous span; else
// (`split` false) every tile is walked once, as on an unfused ring.  Virtual
// tile j goes to CTA rank j % 2.
struct RingWalk {
  bool split = false;
  int cap = 1, nkeys = 0, rows = 0, s0 = 0, count = 0;
  int dbl0 = -1, dbl1 = -1;  // the tiles walked twice, ascending (-1: none)
  __device__ __forceinline__ RingWalk() {}
  __device__ __forceinline__ RingWalk(int cap_, int nkeys_, int past, int rows_, int ntiles) {
    cap = cap_;
    nkeys = nkeys_;
    rows = rows_;
    s0 = past % cap_;
    split = cap_ > kTcBlockN && rows_ <= cap_ - kTcBlockN;
    dbl0 = dbl1 = -1;
    count = ntiles;
    if (split) {
      const int ca = s0 / kTcBlockN, cb = ((s0 + rows - 1) % cap) / kTcBlockN;
      const int c0 = min(ca, cb), c1 = max(ca, cb);
      if (both(c0)) dbl0 = c0;
      if (c1 != c0 && both(c1)) {
        if (dbl0 < 0) dbl0 = c1; else dbl1 = c1;
      }
      count = ntiles + (dbl0 >= 0) + (dbl1 >= 0);
    }
  }
  // The new slots [a, b) of tile t (a == b: none).
  __device__ __forceinline__ void new_span(int t, int& a, int& b) const {
    const int j0 = t * kTcBlockN, j1 = min(j0 + kTcBlockN, nkeys);
    int lo = max(j0, s0), hi = min(j1, min(s0 + rows, cap));
    if (lo < hi) { a = lo; b = hi; return; }
    lo = j0;
    hi = min(j1, s0 + rows - cap);
    if (lo < hi) { a = lo; b = hi; return; }
    a = b = j0;
  }
  __device__ __forceinline__ bool both(int t) const {
    int a, b;
    new_span(t, a, b);
    return a < b && (b - a) < min(t * kTcBlockN + kTcBlockN, nkeys) - t * kTcBlockN;
  }
  __device__ __forceinline__ void at(int w, int& tile, bool& is_new) const {
    int base = 0;  // tiles walked twice before the candidate
    const int d[2] = {dbl0, dbl1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (d[k] < 0) break;
      const int first = d[k] + base;  // walk index of tile d[k]'s cached walk
      if (w < first) break;
      if (w == first || w == first + 1) {
        tile = d[k];
        is_new = w == first + 1;
        return;
      }
      ++base;
    }
    tile = w - base;
    int a, b;
    new_span(tile, a, b);
    is_new = split && a < b;  // a tile walked once holds only new slots or only cached ones
  }
  // Slots [lo, hi) of the tile that hold written data (the interface of Walk;
  // the ring's masks come from the slot-to-position map instead).
  __device__ __forceinline__ void range(int tile, bool, int& lo, int& hi) const {
    lo = tile * kTcBlockN;
    hi = min(lo + kTcBlockN, nkeys);
  }
  // Row of k_new / v_new that slot tile * 128 maps to in a new walk (rows
  // outside [0, rows) are not new slots and read as zero).
  __device__ __forceinline__ int new_row(int tile) const {
    const int j0 = tile * kTcBlockN;
    return j0 - s0 + (j0 + kTcBlockN <= s0 ? cap : 0);
  }
};

// Paged instantiation: whether walk w's K/V stage holds whole pages (the page
// layout) rather than two 128-row boxes read from k_new / v_new.
template <typename W>
__device__ __forceinline__ bool stage_has_pages(const W& walk, int w, int kv_direct, int past) {
  int t;
  bool nw;
  walk.at(w, t, nw);
  return !(kv_direct && t * kTcBlockN >= past);
}

// The walk a kernel instantiation uses: the ring's on a ring cache, else the plain one.
template <bool kRing>
__device__ __forceinline__ const std::conditional_t<kRing, RingWalk, Walk>& pick_walk(const Walk& plain,
                                                                                      const RingWalk& ring) {
  if constexpr (kRing) return ring;
  else return plain;
}

// The last CTA of the grid to take a ticket -- every CTA takes one after all its
// threads have read their sequence's length -- adds commit_add to every length
// and resets the counter for the next launch.  A counter found above the grid
// size was not zero before the launch: reported as CP_DEV_BOUNDS.
__device__ __forceinline__ void take_ticket(const AttnArgs& a) {
  __threadfence();
  const unsigned total = gridDim.x * gridDim.y;
  const unsigned t = atomicAdd(a.ticket, 1u);
  if (t == total - 1) {
    __threadfence();
    for (int q = 0; q < a.rows.num_seqs; ++q) a.commit_lens[q] += a.commit_add;
    __threadfence();
    atomicExch(a.ticket, 0u);
  } else if (t >= total && a.status) {
    atomicOr(a.status, CP_DEV_BOUNDS);
  }
}

template <typename T, int D, bool kRing, bool kPageBox>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ CUtensorMap tm_kn, const __grid_constant__ CUtensorMap tm_vn,
                   const AttnArgs a) {
  using L = TcSmem<D>;
  constexpr int DB = L::DB;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = make_idesc_f16(kBf16, 128, 128, false);
  constexpr uint32_t kIdescPV = make_idesc_f16(kBf16, 128, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::q_off;
  uint8_t* sK = smem + L::k_off;
  uint8_t* sV = smem + L::v_off;
  TcBarriers* bar = reinterpret_cast<TcBarriers*>(smem + L::bar_off);

  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int rpt = kTcBlockM / G;  // tokens per Q tile
  // The cluster's work: with a work list, pair L / hkv of KV head L % hkv for
  // the cluster's linear index L (so the heaviest pairs of every head start
  // first); else pair blockIdx.x / 2 of KV head blockIdx.y.
  const int cl = (int)blockIdx.y * (int)(gridDim.x >> 1) + (int)(blockIdx.x >> 1);
  const int g = a.pair_order ? cl % a.hkv : (int)blockIdx.y;
  const int w_pair = a.pair_order ? cl / a.hkv : (int)(blockIdx.x >> 1);
  const int rank = (int)cluster_ctarank();

  // ---- set-up that reads no global memory: it may overlap the previous kernel
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar->k_full[i], 1);
      mbar_init(&bar->v_full[i], 1);
      mbar_init(&bar->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->q_full[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_ready[i], 128);
    }
    mbar_init(&bar->o_final, 1);
    for (int c = 0; c < L::kMergeChunks; ++c) mbar_init(&bar->merge_full[c], 1);
    mbar_init(&bar->peer_free, 1);
    bar->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    if (a.kv_direct || a.fused) {
      tma_prefetch_desc(&tm_kn);
      tma_prefetch_desc(&tm_vn);
    }
  }
  if (warp == 1) {
    tmem_alloc(&bar->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // barrier inits are visible cluster-wide before any remote access (waited below)
  const uint32_t tmem = bar->tmem_base;
  volatile int* abort_flag = &bar->abort;
  pdl_wait();  // everything below reads what earlier kernels wrote
  if (a.commit_lens && !a.ticket && blockIdx.x == 0 && blockIdx.y == 0)
    for (int q = threadIdx.x; q < a.rows.num_seqs; q += kThreads) a.commit_lens[q] += a.commit_add;

  // ---- this cluster's pair (the same for both CTAs, so both leave together)
  int s = 0, t0 = 0, rows = 0, past = 0;
  bool have_pair = find_pair(a, 2 * rpt, w_pair, s, t0);
  if (have_pair) {
    rows = seq_rows(a.rows, s);
    past = a.past[s];
    if (past < 0 || past + rows > a.max_ctx) {
      if (a.status && threadIdx.x == 0 && rank == 0) atomicOr(a.status, CP_DEV_BOUNDS);
      have_pair = false;
    }
  }
  if (a.ticket) __syncthreads();  // every thread has read its length before this CTA takes a ticket
  if (!have_pair) {
    if (a.ticket && threadIdx.x == 0) take_ticket(a);
    cluster_wait();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }
  const int n = past + rows;  // positions written, including this call's rows
  const int row0 = seq_row0(a.rows, s);
  const int t_end = min(t0 + 2 * rpt, rows);
  // A ring cache: the launcher picks the kRing instantiation for it (compiled
  // for the ring alone); the other instantiation keeps the run-time test.
  const bool rolling = kRing || a.cache.kind == CP_CACHE_ROLLING;
  const bool paged = a.cache.kind == CP_CACHE_PAGED;
  const int cap = a.cache.capacity;
  // Key indices walked: absolute positions [0, nkeys) (contiguous / paged) or
  // physical ring slots [0, nkeys) (rolling).
  const int nkeys = rolling ? min(n, cap) : past + t_end;
  const int n_valid = rolling ? nkeys : n;  // key indices holding written data
  const int ntiles = (nkeys + kTcBlockN - 1) / kTcBlockN;
  const Walk walk_plain(!rolling && !paged, past, n_valid, ntiles);
  const RingWalk walk_ring = kRing ? RingWalk(cap, nkeys, past, rows, ntiles) : RingWalk();
  const auto& walk = pick_walk<kRing>(walk_plain, walk_ring);
  const int nmine = walk.count > rank ? (walk.count - rank + 1) / 2 : 0;  // this CTA's walks: rank + 2i
  const bool q1 = t0 + rpt < rows;  // Q tile 1 holds at least one row (else it is skipped)
  const bool own_tile = rank == 0 || q1;   // Q tile `rank` (finished here) has rows
  const bool peer_tile = rank == 1 || q1;  // Q tile `1 - rank` (finished by the peer) has rows
  const uint32_t peer = (uint32_t)(1 - rank);
  if (threadIdx.x == 0 && own_tile)
    for (int c = 0; c < L::kMergeChunks; ++c)  // chunk 0 also brings the peer's (max, sum)
      mbar_arrive_expect_tx(&bar->merge_full[c], L::kChunkBytes + (c == 0 ? 256u * 4u : 0u));

  if (warp < 4) {
  // The control warpgroup gives up registers for the softmax warpgroups.  Each
  // role keeps to its own branch up to the final cluster barrier, so the
  // compiler holds each branch to its own register budget.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
  if (warp == 0) {
    // ================================================================ producer
    // Issue order Q0, K0, Q1, V0, K1, V1, ...: the first MMA (S0 = Q0 K0^T)
    // waits for 64 KB instead of both Q tiles and the whole first stage.
    auto load_q = [&](int w) {
      mbar_arrive_expect_tx(&bar->q_full[w], DB * kBlockBytes);
      for (int db = 0; db < DB; ++db)
        tma_load_3d(sQ + (w * DB + db) * kBlockBytes, &tm_q, &bar->q_full[w], db * 64, g * G, row0 + t0 + w * rpt);
    };
    if (lane == 0 && nmine > 0) load_q(0);
    const int ps = a.cache.page_size;
    const int npg = paged ? kTcBlockN / ps : 0;
    // One stage = the K tile and the V tile of one KV tile, signalled together.
    int issued = -1;
    for (int i = 0; i < nmine; ++i) {
      const int st = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      int tile;
      bool is_new;
      walk.at(rank + 2 * i, tile, is_new);
      const int j0 = tile * kTcBlockN;
      const bool from_new = a.fused && is_new;  // the call's own rows, read from k_new / v_new
      // A paged tile made only of this call's rows is read from k_new / v_new:
      // two 16 KB boxes per tensor instead of one small box per page.
      const bool direct = paged && a.kv_direct && j0 >= past;
      int my_page = -1;  // paged: lane l looks up the page of keys [j0 + l*ps, ...)
      if (paged && !direct && lane < npg) {
        const int key = j0 + lane * ps;
        if (key < n_valid) {
          const int blk = key / ps;
          if (blk < a.cache.max_blocks) my_page = a.cache.block_table[(long long)s * a.cache.max_blocks + blk];
          if (my_page < 0 || my_page >= a.cache.num_pages) {
            if (a.status) atomicOr(a.status, CP_DEV_BOUNDS);
            my_page = -1;
          }
        }
      }
      const uint32_t page_mask = paged ? __ballot_sync(0xffffffffu, my_page >= 0) : 0u;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&bar->kv_empty[st], ph ^ 1, abort_flag, a.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint64_t* kf = &bar->k_full[st];
      uint64_t* vf = &bar->v_full[st];
      uint8_t* dk = sK + st * DB * kBlockBytes;
      uint8_t* dv = sV + st * DB * kBlockBytes;
      if (from_new) {
        // Fused append: keys [j0, j0 + 128) are rows j0 - past ... of this
        // sequence's k_new / v_new (4-D maps: rows outside [0, rows) read as zero).
        if constexpr (kRing) {
          // On a ring, slot j0 maps to row walk.new_row(tile).
          if (lane == 0) {
            const int nr = walk.new_row(tile);
            mbar_arrive_expect_tx(kf, DB * kBlockBytes);
            for (int db = 0; db < DB; ++db) tma_load_4d(dk + db * kBlockBytes, &tm_kn, kf, db * 64, g, nr, s);
            if (i == 0 && q1) load_q(1);
            mbar_arrive_expect_tx(vf, DB * kBlockBytes);
            for (int db = 0; db < DB; ++db) tma_load_4d(dv + db * kBlockBytes, &tm_vn, vf, db * 64, g, nr, s);
          }
        } else {
        if (lane == 0) {
          mbar_arrive_expect_tx(kf, DB * kBlockBytes);
          for (int db = 0; db < DB; ++db) tma_load_4d(dk + db * kBlockBytes, &tm_kn, kf, db * 64, g, j0 - past, s);
          if (i == 0 && q1) load_q(1);
          mbar_arrive_expect_tx(vf, DB * kBlockBytes);
          for (int db = 0; db < DB; ++db) tma_load_4d(dv + db * kBlockBytes, &tm_vn, vf, db * 64, g, j0 - past, s);
        }
        }
      } else if (!paged || direct) {
        // Contiguous: keys [j0, j0 + 128) of KV head g.  Direct: they are rows
        // row0 + (j0 - past) ... of k_new / v_new (rows past this sequence's
        // are masked, and zeroed in the last V tile).
        if (lane == 0) {
          const CUtensorMap* mk = direct ? &tm_kn : &tm_k;
          const CUtensorMap* mv = direct ? &tm_vn : &tm_v;
          const int c1 = direct ? g : j0;
          const int c2 = direct ? row0 + (j0 - past) : s * a.hkv + g;
          mbar_arrive_expect_tx(kf, DB * kBlockBytes);
          for (int db = 0; db < DB; ++db) tma_load_3d(dk + db * kBlockBytes, mk, kf, db * 64, c1, c2);
          if (i == 0 && q1) load_q(1);
          mbar_arrive_expect_tx(vf, DB * kBlockBytes);
          for (int db = 0; db < DB; ++db) tma_load_3d(dv + db * kBlockBytes, mv, vf, db * 64, c1, c2);
        }
      } else {
        const uint32_t bytes = (uint32_t)__popc(page_mask) * DB * ps * 128u;
        if (lane == 0) {
          mbar_arrive_expect_tx(kf, bytes);
          mbar_arrive_expect_tx(vf, bytes);
        }
        __syncwarp();
        if constexpr (kPageBox) {
          // One box per page and lane, both 64-column halves: page pi lands at
          // pi * ps * 256 as 8-row groups [ps / 8][half][8 rows][128 B] (the
          // page layout); lanes npg .. 2 npg - 1 load V.
          const int pi = lane % npg;
          const int page = __shfl_sync(0xffffffffu, my_page, pi);
          if (lane < 2 * npg && page >= 0) {
            const bool is_v = lane >= npg;
            tma_load_4d((is_v ? dv : dk) + pi * ps * 256, is_v ? &tm_v : &tm_k, is_v ? vf : kf, 0, 0, 0,
                        (page * a.hkv + g) * (ps / 8));
          }
        } else {
        // One box per lane: box b < 2 * npg * DB is tensor b / (npg * DB) (K, then V),
        // page (b / DB) % npg, 64-column half b % DB.
        const int nbox = npg * DB;
        for (int b0 = 0; b0 < 2 * nbox; b0 += 32) {
          const int b = b0 + lane;
          const int pi = (b / DB) % npg;
          const int page = __shfl_sync(0xffffffffu, my_page, pi);
          if (b < 2 * nbox && page >= 0) {
            const bool is_v = b >= nbox;
            const int db = b % DB;
            tma_load_3d((is_v ? dv : dk) + db * kBlockBytes + pi * ps * 128, is_v ? &tm_v : &tm_k, is_v ? vf : kf,
                        db * 64, 0, page * a.hkv + g);
          }
        }
        }
        if (lane == 0 && i == 0 && q1) load_q(1);
      }
      issued = i;
    }
    if (lane == 0 && *abort_flag) {
      // Let copies already in flight land before the CTA's shared memory is released.
      volatile int zero = 0;
      if (nmine > 0) mbar_wait(&bar->q_full[0], 0, &zero, nullptr);
      if (q1 && issued >= 0) mbar_wait(&bar->q_full[1], 0, &zero, nullptr);
      for (int t = issued - 1; t <= issued; ++t)
        if (t >= 0) {
          mbar_wait(&bar->k_full[t & 1], (t >> 1) & 1, &zero, nullptr);
          mbar_wait(&bar->v_full[t & 1], (t >> 1) & 1, &zero, nullptr);
        }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // The whole warp runs the loop, converged; one elected lane issues each
    // tcgen05 instruction (operands stay warp-uniform, so MMAs issue back to
    // back).  Per KV tile four waits (P0, V, K of the next tile, P1) and three
    // commits.
    {
      auto wait = [&](uint64_t* b, uint32_t parity) { return warp_wait(b, parity, abort_flag, a.status); };
      constexpr uint64_t kTileStep = (DB * kBlockBytes) >> 4;
      const uint64_t q_desc0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(sV), kBlockBytes, 1024);
      // Page layout (the paged instantiation's page boxes): K's 8-row groups
      // 2048 B apart with the second 64-column half 1024 B in; V's 16-key steps
      // 4096 B apart, its 8-key groups 2048 B and its halves (the MMA's N
      // blocks) 1024 B apart.  Tiles read from k_new keep the two-box layout.
      auto issue_qk = [&](int w, int i) {  // S_w = Q_w K_i^T
        if constexpr (kPageBox) {
          const bool pg = stage_has_pages(walk, rank + 2 * i, a.kv_direct, past);
          const uint64_t q_desc = q_desc0 + w * kTileStep;
          const uint64_t k_desc = (pg ? make_sdesc_sw128(smem_u32(sK), 16, 2048) : k_desc0) + (i & 1) * kTileStep;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = ((kk >> 2) * kBlockBytes + (kk & 3) * 32) >> 4;
            const uint64_t koff = pg ? ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4 : off;
            mma_ss_elect(tmem + 256u * w, q_desc + off, k_desc + koff, kIdescQK, kk > 0);
          }
          mma_commit_elect(&bar->s_full[w]);
        } else {
        const uint64_t q_desc = q_desc0 + w * kTileStep;
        const uint64_t k_desc = k_desc0 + (i & 1) * kTileStep;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * kBlockBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem + 256u * w, q_desc + off, k_desc + off, kIdescQK, kk > 0);
        }
        mma_commit_elect(&bar->s_full[w]);
        }
      };
      auto issue_pv = [&](int w, int i) {  // O_w += P_w V_i
        if constexpr (kPageBox) {
          const bool pg = stage_has_pages(walk, rank + 2 * i, a.kv_direct, past);
          const uint64_t v_desc = (pg ? make_sdesc_sw128(smem_u32(sV), 1024, 2048) : v_desc0) + (i & 1) * kTileStep;
          const int step = pg ? 4096 : 2048;
#pragma unroll
          for (int kk = 0; kk < kTcBlockN / 16; ++kk)
            mma_ts_elect(tmem + 256u * w + 128u, tmem + 256u * w + kk * 8, v_desc + ((kk * step) >> 4), kIdescPV,
                         (i > 0 || kk > 0) ? 1u : 0u);
        } else {
        const uint64_t v_desc = v_desc0 + (i & 1) * kTileStep;
#pragma unroll
        for (int kk = 0; kk < kTcBlockN / 16; ++kk)
          mma_ts_elect(tmem + 256u * w + 128u, tmem + 256u * w + kk * 8, v_desc + ((kk * 2048) >> 4), kIdescPV,
                       (i > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = nmine > 0 && wait(&bar->q_full[0], 0) && wait(&bar->k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
      }
      if (ok && q1) {
        ok = wait(&bar->q_full[1], 0);
        if (ok) {
          tc_fence_after();
          issue_qk(1, 0);
        }
      }
      for (int i = 0; ok && i < nmine; ++i) {
        const bool more = i + 1 < nmine;
        if (!wait(&bar->p_ready[0], i & 1)) break;
        if (!wait(&bar->v_full[i & 1], (i >> 1) & 1)) break;
        int ztile;
        bool znew;
        walk.at(rank + 2 * i, ztile, znew);
        if constexpr (kRing) {
          if (!(a.fused && znew)) {  // read from the ring: zero V rows that hold no slot of this walk
            uint8_t* v_stage = sV + (i & 1) * DB * kBlockBytes;
            auto zero_rows = [&](int lo, int hi) {  // rows [lo, hi) of the tile
              const int nvec = max(hi - lo, 0) * 128 / 16;
              for (int db = 0; db < DB; ++db) {
                uint4* p = reinterpret_cast<uint4*>(v_stage + db * kBlockBytes + lo * 128);
                for (int e = lane; e < nvec; e += 32) p[e] = make_uint4(0, 0, 0, 0);
              }
            };
            const int jz = ztile * kTcBlockN;
            const int valid = min(jz + kTcBlockN, walk.nkeys) - jz;  // rows holding written slots
            int na, nb;
            walk.new_span(ztile, na, nb);
            if (!walk.split) {
              zero_rows(valid, kTcBlockN);
            } else if (znew) {  // keep the new span only
              zero_rows(0, na - jz);
              zero_rows(nb - jz, kTcBlockN);
            } else {  // keep the cached slots: zero the new span and the unwritten tail
              zero_rows(na - jz, nb - jz);
              zero_rows(valid, kTcBlockN);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        } else {
        if (!(a.fused && znew)) {  // read from the cache: zero V rows that hold no key of this walk
          int zlo, zhi;
          walk.range(ztile, znew, zlo, zhi);
          const int tail = max(zhi - ztile * kTcBlockN, 0);
          if (tail < kTcBlockN) {
            uint8_t* v_stage = sV + (i & 1) * DB * kBlockBytes;
            const int nvec = (kTcBlockN - tail) * 128 / 16;
            if constexpr (kPageBox) {
              // Page layout: row r of half db at (r / 8) * 2048 + db * 1024 + (r % 8) * 128.
              if (stage_has_pages(walk, rank + 2 * i, a.kv_direct, past)) {
                for (int e = lane; e < nvec * DB; e += 32) {
                  const int r = tail + e / (8 * DB), db = (e / 8) % DB;
                  *reinterpret_cast<uint4*>(v_stage + (r >> 3) * 2048 + db * 1024 + (r & 7) * 128 + (e & 7) * 16) =
                      make_uint4(0, 0, 0, 0);
                }
              } else {
                for (int db = 0; db < DB; ++db) {
                  uint4* p = reinterpret_cast<uint4*>(v_stage + db * kBlockBytes + tail * 128);
                  for (int e = lane; e < nvec; e += 32) p[e] = make_uint4(0, 0, 0, 0);
                }
              }
            } else {
            for (int db = 0; db < DB; ++db) {
              uint4* p = reinterpret_cast<uint4*>(v_stage + db * kBlockBytes + tail * 128);
              for (int e = lane; e < nvec; e += 32) p[e] = make_uint4(0, 0, 0, 0);
            }
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        }
        tc_fence_after();
        issue_pv(0, i);
        if (more) {
          if (!wait(&bar->k_full[(i + 1) & 1], ((i + 1) >> 1) & 1)) break;
          issue_qk(0, i + 1);
        }
        if (q1) {
          if (!wait(&bar->p_ready[1], i & 1)) break;
          tc_fence_after();
          issue_pv(1, i);
        }
        mma_commit_elect(&bar->kv_empty[i & 1]);
        if (more && q1) issue_qk(1, i + 1);
      }
      // o_final: every MMA issued has completed (epilogue and TMEM release wait on it).
      mma_commit_elect(&bar->o_final);
      volatile int zero = 0;  // wait even after an abort: MMAs may still be in flight
      mbar_wait(&bar->o_final, 0, &zero, a.status);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ================================================================ fused append
    // The K/V rows of Q tile `rank`'s tokens for KV head g go to their slots
    // past + t of the cache ([Wiki] 一.1); every (token, KV head) row of the
    // chunk belongs to exactly one Q tile.  No tile of this launch reads them
    // from the cache: the walks that hold them read k_new / v_new.
    if (a.fused) {
      const int tk0 = t0 + rank * rpt, tk1 = min(tk0 + rpt, rows);
      const int nrow = max(tk1 - tk0, 0);
      constexpr int kVec = D * 2 / 16;  // 16-byte vectors per row
      const long long src_row = (long long)row0 + tk0;
      const long long dst_row = ((long long)(s * a.hkv + g)) * cap + past + tk0;
      if constexpr (kRing) {
        for (int e = lane; e < nrow * kVec; e += 32) {  // position past + t lives in slot (past + t) mod cap
          const int r = e / kVec, c = e % kVec;
          const long long so = ((src_row + r) * a.hkv + g) * kVec + c;
          const long long dof = (((long long)(s * a.hkv + g)) * cap + (past + tk0 + r) % cap) * kVec + c;
          const uint4 kv = reinterpret_cast<const uint4*>(a.k_new)[so];
          const uint4 vv = reinterpret_cast<const uint4*>(a.v_new)[so];
          reinterpret_cast<uint4*>(a.k_cache)[dof] = kv;
          reinterpret_cast<uint4*>(a.v_cache)[dof] = vv;
        }
      } else {
      for (int e = lane; e < nrow * kVec; e += 32) {
        const int r = e / kVec, c = e % kVec;
        const long long so = ((src_row + r) * a.hkv + g) * kVec + c;
        const long long dof = (dst_row + r) * kVec + c;
        const uint4 kv = reinterpret_cast<const uint4*>(a.k_new)[so];
        const uint4 vv = reinterpret_cast<const uint4*>(a.v_new)[so];
        reinterpret_cast<uint4*>(a.k_cache)[dof] = kv;
        reinterpret_cast<uint4*>(a.v_cache)[dof] = vv;
      }
      }
    }
  } else if (warp == 3) {
    // Every thread of this CTA has read its length (the __syncthreads after the
    // lookup); the last CTA to take a ticket advances them all.
    if (a.ticket && lane == 0) take_ticket(a);
  }
  cluster_wait();  // the peer's barriers are initialised
  if (warp == 1 && lane == 0 && own_tile) {
    // This CTA's MMAs are complete (the issuer waited o_final): its K/V stages are free.
    mbar_arrive_remote(mapa_shared(smem_u32(&bar->peer_free), peer));
  }
  } else {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
  // ================================================================ softmax groups
  const int grp = (warp - 4) >> 2;          // Q tile of this group
  const int quarter = warp & 3;             // TMEM lanes [32*quarter, +32)
  const int mrow = quarter * 32 + lane;     // this thread's row of its Q tile
  const int tok = t0 + grp * rpt + mrow / G;
  const int head = g * G + mrow % G;
  const bool row_ok = tok < t_end;
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const uint32_t s_col = tmem + lane_off + 256u * grp;
  const uint32_t o_col = s_col + 128u;
  float m_run = -INFINITY;  // max used for exponentiation (log2 domain)
  float l_run = 0.f;
  bool alive = true;
  if (grp == 0 || q1) {
    const int p_row = row_ok ? past + tok : -1;  // absolute query position
    const int lo = rolling ? max(a.left_pad ? a.left_pad[s] : 0, 0) : 0;
    // Rolling: slot -> absolute position (see cp_kv.cuh), split at slot r_slot.
    const int r_slot = n > 0 ? (n - 1) % cap : 0;
    const int base_hi = n - 1 - r_slot;
    const float sl2 = a.scale_log2;
    for (int i = 0; i < nmine; ++i) {
      if (!warp_wait(&bar->s_full[grp], i & 1, abort_flag, a.status)) { alive = false; break; }
      tc_fence_after();
      uint32_t sv[128];
      tmem_ld32(s_col + 0, &sv[0]);
      tmem_ld32(s_col + 32, &sv[32]);
      tmem_ld32(s_col + 64, &sv[64]);
      tmem_ld32(s_col + 96, &sv[96]);
      tmem_wait_ld();
      int tile;
      bool is_new;
      walk.at(rank + 2 * i, tile, is_new);
      const int j0 = tile * kTcBlockN;
      float mx = -INFINITY;
      if (!rolling) {
        // Visible columns [c_lo, c_hi): keys of this walk at or before the row.
        int klo, khi;
        walk.range(tile, is_new, klo, khi);
        const int c_lo = klo - j0, c_hi = min(khi, p_row + 1) - j0;
        if (c_lo > 0 || c_hi < kTcBlockN) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < c_lo || c >= c_hi) sv[c] = __float_as_uint(-INFINITY);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = j0 + c;
          const int pos = key + base_hi - (key > r_slot ? cap : 0);
          const bool vis = key < nkeys && pos >= lo && pos <= p_row;
          if (!vis) sv[c] = __float_as_uint(-INFINITY);
        }
        if constexpr (kRing) {
          if (tile == walk.dbl0 || tile == walk.dbl1) {  // walked twice: this walk's slots only
            int na, nb;
            walk.new_span(tile, na, nb);
            const int ca = na - j0, cb = nb - j0;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if ((c >= ca && c < cb) != is_new) sv[c] = __float_as_uint(-INFINITY);
          }
        }
      }
      {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          m4[0] = fmax3(m4[0], __uint_as_float(sv[c + 0]), __uint_as_float(sv[c + 1]));
          m4[1] = fmax3(m4[1], __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
          m4[2] = fmax3(m4[2], __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
          m4[3] = fmax3(m4[3], __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
        }
        mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      }
      const float mx2 = mx * sl2;  // scale > 0, so the max commutes with it
      const bool grow = mx2 > m_run + kRescaleLog2 || (m_run == -INFINITY && mx2 != -INFINITY);
      const float m_new = grow ? mx2 : m_run;
      const float alpha = grow ? (m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new)) : 1.f;
      const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float x0 = __uint_as_float(sv[2 * c]), x1 = __uint_as_float(sv[2 * c + 1]);
        ffma2(x0, x1, sl2, neg_m);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        fadd2(ps4[2 * (c & 1)], ps4[2 * (c & 1) + 1], p0, p1);
        sv[c] = pack2<T>(p0, p1);
      }
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      l_run = l_run * alpha + psum;
      m_run = m_new;
      tmem_st32(s_col + 0, &sv[0]);
      tmem_st32(s_col + 32, &sv[32]);
      // O holds P V of this group's earlier tiles (complete: see the ordering
      // note above).  Rows whose max grew rescale it; the others multiply by 1.
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_col + 32 * c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(o_col + 32 * c, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->p_ready[grp]);
    }
  }

  // ================================================================ merge across the pair
  volatile int zero = 0;
  const bool done = warp_wait(&bar->o_final, 0, &zero, a.status) && alive;
  tc_fence_after();
  __syncwarp();
  cluster_wait();  // the peer's barriers are initialised
  const bool have_o = nmine > 0;  // this CTA wrote O (else its TMEM O is unset: send zeros)
  if (grp != rank && peer_tile) {
    // Rows of Q tile (1 - rank) are finished by the peer: stage this CTA's
    // partial one 32-column chunk at a time and send each chunk as soon as it
    // is staged, so one chunk's transfer overlaps the staging of the next.
    bar->out_ml[mrow] = have_o ? m_run : -INFINITY;
    bar->out_ml[128 + mrow] = have_o ? l_run : 0.f;
    bool send = true;  // (meaningful in the thread of row 0, which sends)
#pragma unroll
    for (int c = 0; c < L::kMergeChunks; ++c) {
      uint32_t ov[32];
      if (have_o) {
        tmem_ld32(o_col + 32 * c, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<uint4*>(sK + merge_off(mrow, c, e)) =
            make_uint4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
      fence_proxy_async_smem();  // the bulk copy reads these through the async proxy
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (mrow == 0) {
        if (c == 0) send = mbar_wait_cluster(&bar->peer_free, 0, a.status);
        if (send) {
          const uint32_t rbar = mapa_shared(smem_u32(&bar->merge_full[c]), peer);
          bulk_copy_to_peer(mapa_shared(smem_u32(sV + c * L::kChunkBytes), peer), sK + c * L::kChunkBytes,
                            L::kChunkBytes, rbar);
          if (c == 0) bulk_copy_to_peer(mapa_shared(smem_u32(bar->peer_ml), peer), bar->out_ml, 256u * 4u, rbar);
        }
      }
    }
  }
  if (grp == rank && own_tile) {
    // Fixed order: the even-tile half (rank 0's partial) first.  Chunk 0
    // brings the peer's (max, sum); each chunk is combined as it lands.
    bool got = mbar_wait_cluster(&bar->merge_full[0], 0, a.status);
    const float m_own = have_o ? m_run : -INFINITY, l_own = have_o ? l_run : 0.f;
    const float m_peer = bar->peer_ml[mrow], l_peer = bar->peer_ml[128 + mrow];
    const float mA = rank == 0 ? m_own : m_peer, lA = rank == 0 ? l_own : l_peer;
    const float mB = rank == 0 ? m_peer : m_own, lB = rank == 0 ? l_peer : l_own;
    const float mm = fmaxf(mA, mB);
    const float wA = (mA == -INFINITY) ? 0.f : ex2_approx(mA - mm);
    const float wB = (mB == -INFINITY) ? 0.f : ex2_approx(mB - mm);
    const float lsum = lA * wA + lB * wB;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    // A tile whose rows all belong to this sequence leaves through a TMA store
    // from the (now unused) Q buffer; a ragged tile row by row.
    const int tile_tok0 = t0 + rank * rpt;
    const bool full_tile = tile_tok0 + rpt <= t_end;
    uint8_t* sOut = sQ + rank * DB * kBlockBytes;
    T* out = static_cast<T*>(a.out) + ((long long)(row0 + tok) * a.hq + head) * D;
#pragma unroll
    for (int c = 0; c < L::kMergeChunks; ++c) {
      if (c > 0 && got) got = mbar_wait_cluster(&bar->merge_full[c], 0, a.status);
      uint32_t ov[32];
      if (have_o) {
        tmem_ld32(o_col + 32 * c, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 pr = *reinterpret_cast<const float4*>(sV + merge_off(mrow, c, e));
        const float own[4] = {__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                              __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3])};
        const float prv[4] = {pr.x, pr.y, pr.z, pr.w};
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = rank == 0 ? own[u] * wA + prv[u] * wB : prv[u] * wA + own[u] * wB;
        pk[2 * e] = pack2<T>(x[0] * inv, x[1] * inv);
        pk[2 * e + 1] = pack2<T>(x[2] * inv, x[3] * inv);
      }
      if (full_tile) {
        // Columns [32c, 32c + 32) are 16-byte chunks 4(c%2) .. 4(c%2)+3 of box c/2 (128B swizzle).
        uint8_t* box = sOut + (c >> 1) * kBlockBytes + mrow * 128;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int chunk = (c & 1) * 4 + e;
          *reinterpret_cast<uint4*>(box + ((chunk ^ (mrow & 7)) * 16)) =
              make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      } else if (done && got && row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
    if (full_tile) {
      fence_proxy_async_smem();  // the TMA store reads the tile through the async proxy
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (mrow == 0 && done && got) {
        for (int db = 0; db < DB; ++db)
          tma_store_3d(&tm_o, sOut + db * kBlockBytes, db * 64, g * G, row0 + tile_tok0);
        bulk_commit_group();
        bulk_wait_read_all();  // the Q buffer is read out; the writes finish with the grid
      }
    }
  }
  }  // softmax warpgroups

  // Both CTAs leave together: the copies each sent into the other have landed
  // and been read before either CTA's shared memory is released.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D, bool kRing, bool kPageBox = false>
cudaError_t launch_t(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& to, const CUtensorMap& tkn, const CUtensorMap& tvn, int pairs_bound,
                     cudaStream_t st) {
  // D = 64 would fit two CTAs per SM, but each CTA takes all 512 TMEM
  // columns; ask for enough shared memory to keep it at one CTA per SM.
  const uint32_t smem = TcSmem<D>::alloc < 120u * 1024u ? 120u * 1024u : TcSmem<D>::alloc;
  // Raise the dynamic shared-memory limit once per device (it is a per-device
  // function attribute), so later calls -- including ones being captured into
  // a CUDA graph -- only launch.
  static std::atomic<uint64_t> ready_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready_mask.load(std::memory_order_acquire) & bit)) {
    // The register split is only sound at the per-thread count it was sized
    // for: refuse to launch a build that came out at another count.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_tc_kernel<T, D, kRing, kPageBox>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(attn_tc_kernel<T, D, kRing, kPageBox>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ready_mask.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: set-up overlaps the previous kernel (see launch_pdl).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * pairs_bound, a.hkv);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<T, D, kRing, kPageBox>, tq, tk, tv, to, tkn, tvn, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(int d, int group, int dtype) {
  return (d == 64 || d == 128) && group >= 1 && group <= 16 && (group & (group - 1)) == 0 &&
         (dtype == CP_BF16 || dtype == CP_F16);
}

// pairs_bound: number of 2*128-row Q-tile pairs to cover (one 2-CTA cluster each).
// to: the output [rows, Hq, D] with the same box as tq (finished tiles are TMA-stored).
// tk, tv on a paged cache with D = 128: page-row maps (make_tc_maps), one box per page.
// tkn, tvn: this call's new K/V rows: [rows, Hkv, D] with box {64, 1, 128} when a.kv_direct
// (paged), [num_seqs, rows_uniform, Hkv, D] with box {64, 1, 128, 1} when a.fused (contiguous).
cudaError_t launch_attn_tc(const AttnArgs& a, int dtype, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const CUtensorMap& tkn,
                           const CUtensorMap& tvn, int pairs_bound, cudaStream_t st) {
  if (pairs_bound <= 0) return cudaSuccess;
  const bool ring = a.cache.kind == CP_CACHE_ROLLING;
  if (a.cache.kind == CP_CACHE_PAGED && a.d == 128)  // page-layout stages (tk, tv: page-row maps)
    return dtype == CP_BF16 ? launch_t<__nv_bfloat16, 128, false, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st)
                            : launch_t<__half, 128, false, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st);
  if (dtype == CP_BF16) {
    if (ring)
      return a.d == 64 ? launch_t<__nv_bfloat16, 64, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st)
                       : launch_t<__nv_bfloat16, 128, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st);
    return a.d == 64 ? launch_t<__nv_bfloat16, 64, false>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st)
                     : launch_t<__nv_bfloat16, 128, false>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st);
  }
  if (ring)
    return a.d == 64 ? launch_t<__half, 64, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st)
                     : launch_t<__half, 128, true>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st);
  return a.d == 64 ? launch_t<__half, 64, false>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st)
                   : launch_t<__half, 128, false>(a, tq, tk, tv, to, tkn, tvn, pairs_bound, st);
}

}  // namespace cp
