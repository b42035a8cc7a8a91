// attn_pair.cu -- chunk attention on paired SMs (tcgen05 cta_group::2), head_dim 128.
//
// What it computes ([Wiki] 一.2; [Glossary] "How chunked prefill works"): row i
// of a chunk is the query at absolute position p = past + i and attends to the
// keys at positions [0, p] -- the cached prefix plus its own causal triangle --
// over a cache bound at fixed physical capacity whose valid length is
// seqlens_k ([Wiki] 一.3).  With the fused append it also writes the chunk's
// K/V rows into the cache ([Wiki] 一.1: chunk k writes only its own slots) and
// advances seqlens_k by the real rows ([Wiki] 四).
//
// Work decomposition.  GroupQueryAttention packs the G = Hq/Hkv query heads of
// one KV head into 128-row Q tiles: 128/G consecutive tokens x G heads, row
// m <-> (token m / G, head m % G).  A cluster of two CTAs on two SMs owns two
// consecutive Q tiles, one per CTA, and both walk the same KV tiles (128 keys,
// aligned to absolute key 0) as one M=256 MMA unit: one thread of CTA 0 issues
//   S = Q K^T   (A: each CTA's own Q tile; B: keys [64r, 64r+64) of the tile
//               in CTA r's shared memory),
//   O += P V    (A: P in each CTA's TMEM; B: head dims [64r, 64r+64) of the
//               tile's V rows in CTA r's shared memory),
// so each SM receives half of every K/V tile and computes its own 128 rows.
// No partial results cross the pair: each CTA finishes its own Q tile.
//
// Tiles that hold keys of this call's chunk (positions >= past) are read from
// k_new / v_new when the append is fused; a tile that straddles `past` is
// walked twice, once per source, each time with only its own keys visible.
// The split at `past` is made whether or not the append is fused, so the fused
// and the separate-call paths do identical arithmetic; padded and unpadded
// runs of the same rows do too (tiles are aligned to absolute positions and
// extra tiles only hold keys that real rows do not see).
//
// Warp roles (384 threads, three warpgroups):
//   warp 0      TMA producer: this CTA's Q tile (issued right after the
//               dependency wait), then per KV tile its K half and V half into a
//               5-stage ring.
//   warp 1      TMEM allocation (both CTAs); in CTA 0 the issuer of S = Q K^T
//               (the whole warp, one elected lane issuing).
//   warp 2      forwarder: when a stage lands in this CTA it zeroes V rows that
//               hold no key of the tile's source (so 0 * stale data never reaches
//               O) and tells CTA 0's issuer (local or remote mbarrier arrive).
//   warp 3      fused append: copies this Q tile's tokens' K/V rows of the
//               KV head into the cache with 16-byte loads and stores; then, in
//               CTA 0, the issuer of O += P V.
//   warps 4-11  softmax: warps 4-7 take the even tiles, warps 8-11 the odd ones;
//               thread (warp, lane) owns row 32*(warp%4) + lane and all 128 keys
//               of its tiles.  The running max of a row is handed from one
//               warpgroup to the other through shared memory after each tile's
//               row max, so one warpgroup exponentiates while the other loads
//               and reduces the next tile; each keeps its own share of the row
//               sum and the two are added at the end.
// TMEM (512 columns): S double buffer [0,128) and [128,256), P double buffer
// [256,320) and [320,384) (16-bit pairs), O [384,512).  P has its own columns,
// so S of tile i+2 is computed as soon as the softmax has read S of tile i
// (into registers), while P of tile i still waits for its P V.
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

constexpr int kPThreads = 384;
// Register split: compiled at kPRegsLaunch per thread (the most 384 threads may
// have at one CTA per SM); the control warpgroup (warps 0-3) then drops to
// kPRegsControl and hands the rest to the two softmax warpgroups.
constexpr int kPRegsLaunch = 168;
constexpr int kPRegsControl = 104;
constexpr int kPRegsSoftmax = 200;
static_assert(128 * kPRegsControl + 256 * kPRegsSoftmax == kPThreads * kPRegsLaunch, "the split must add up");
constexpr int kPStages = 5;
constexpr uint32_t kQBlock = 128u * 128u;     // [128 rows][64 x 16-bit]: one 64-dim block of the Q tile
constexpr uint32_t kKHalfBlock = 64u * 128u;  // [64 keys][64 x 16-bit]: one 64-dim block of a K half
constexpr uint32_t kVOff = 2u * kKHalfBlock;  // V half after the two K-half blocks of a stage
constexpr uint32_t kStageBytes = kVOff + kQBlock;  // K half 16 KB + V half [128 keys][64 dims] 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 2;
constexpr int kORing = 8;  // slots of the "P V of tile t done" barrier ring
constexpr uint32_t kColP = 256;  // P of buffer b at kColP + 64 b
constexpr uint32_t kColO = 384;
constexpr float kRescaleLog2 = 8.0f;  // O is rescaled when a row's max grows by more than 2^8

struct __align__(16) PairBarriers {
  uint64_t q_full;               // this CTA's Q tile landed
  uint64_t kv_full[kPStages];    // this CTA's halves of a stage landed
  uint64_t kv_empty[kPStages];   // the stage's MMAs completed (issuer, multicast to both CTAs)
  uint64_t q_ready;              // CTA 0: both Q tiles landed (2 forwarders)
  uint64_t kv_ready[kPStages];   // CTA 0: both CTAs' halves of the stage are ready (2 forwarders)
  uint64_t s_full[kSBufs];       // S buffer b holds its tile's scores (multicast)
  uint64_t s_free[kSBufs];       // CTA 0: S buffer b read out in both CTAs (the tile's 4 warps in each)
  uint64_t p_ready[kSBufs];      // CTA 0: P buffer b written in both CTAs (the tile's 4 warps in each)
  uint64_t o_done[kORing];       // P V of tile t completed, in slot t % kORing (multicast)
  uint64_t qk_final;             // CTA 0: every S MMA issued has completed
  uint64_t o_final;              // every MMA issued has completed (multicast, once)
  uint32_t tmem_base;
  int abort;
  int s, t0, rows, past, have;   // this cluster's pair, read once after the dependency wait
  int q_issued;                  // the Q tile's load was issued
  float xmax[2][2][128];         // [warpgroup][0: running max handed on, 1: last max used][row]
  float xsum[2][128];            // [warpgroup][row] share of the row sum, exchanged at the end
};

struct PairSmem {
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t stage_off = 2 * kQBlock;
  static constexpr uint32_t bar_off = stage_off + kPStages * kStageBytes;
  static constexpr uint32_t bytes = bar_off + sizeof(PairBarriers);
  static constexpr uint32_t alloc = bytes + 1024;  // slack for 1024-byte alignment
};

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

// The KV tiles a pair walks.  Absolute tile t holds keys [128t, 128t + 128).
// Tiles entirely below `past` hold cached keys, tiles entirely at or above it
// the chunk's own keys; a tile that straddles `past` is walked twice (its cached
// keys, then its new ones), so virtual tile j maps to (tile, from_new).
struct TilePlan {
  int past, n, ntiles, tp;
  bool straddle;
  int count;  // virtual tiles

  __device__ __forceinline__ TilePlan(int past_, int rows, int t_end) {
    past = past_;
    n = past_ + rows;
    ntiles = (past_ + t_end + 127) / 128;  // keys visible to the pair's last row
    tp = past_ / 128;
    straddle = (past_ & 127) != 0;
    count = ntiles + (straddle ? 1 : 0);
  }
  __device__ __forceinline__ void at(int j, int& tile, bool& is_new) const {
    if (j < tp) {
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
  // Keys [lo, hi) of the tile that belong to this walk.
  __device__ __forceinline__ void range(int tile, bool is_new, int& lo, int& hi) const {
    const int j0 = tile * 128;
    lo = is_new ? max(j0, past) : j0;
    hi = is_new ? min(j0 + 128, n) : min(j0 + 128, past);
  }
};

// The same with the light remote arrive (the data the waiter needs travels
// through the tensor core, ordered by tcgen05 fences around the arrive).
__device__ __forceinline__ void arrive_leader_light(uint64_t* bar, int rank) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_remote_light(mapa_shared(smem_u32(bar), 0));
}

__device__ __forceinline__ void arrive_leader(uint64_t* bar, int rank) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
}

// The last CTA of the grid to take a ticket -- every CTA takes one after it
// has read its sequence's length -- adds commit_add to every length and resets
// the counter for the next launch.  A counter found above the grid size was not
// zero before the launch: reported as CP_DEV_BOUNDS, nothing is advanced.
__device__ __forceinline__ void take_ticket(const PairArgs& a) {
  if (!a.commit_lens) return;
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

template <typename T>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_vh,
                     const __grid_constant__ CUtensorMap tm_knh, const __grid_constant__ CUtensorMap tm_vnh,
                     const PairArgs a) {
  constexpr int D = 128;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdescQK = make_idesc_f16(kBf16, 256, 128, false);
  constexpr uint32_t kIdescPV = make_idesc_f16(kBf16, 256, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + PairSmem::q_off;
  uint8_t* sStage = smem + PairSmem::stage_off;
  PairBarriers* bar = reinterpret_cast<PairBarriers*>(smem + PairSmem::bar_off);

  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int rpt = 128 / G;  // tokens per Q tile
  const int g = blockIdx.y;
  const int rank = (int)cluster_ctarank();

  // ---- set-up that reads no global memory: it may overlap the previous kernel
  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_ready, 2);
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&bar->kv_full[i], 1);
      mbar_init(&bar->kv_empty[i], 1);
      mbar_init(&bar->kv_ready[i], 2);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&bar->s_full[b], 1);
      mbar_init(&bar->s_free[b], 8);
      mbar_init(&bar->p_ready[b], 8);
    }
    for (int t = 0; t < kORing; ++t) mbar_init(&bar->o_done[t], 1);
    mbar_init(&bar->qk_final, 1);
    mbar_init(&bar->o_final, 1);
    bar->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_o);
    tma_prefetch_desc(&tm_kh);
    tma_prefetch_desc(&tm_vh);
    if (a.fused) {
      tma_prefetch_desc(&tm_knh);
      tma_prefetch_desc(&tm_vnh);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&bar->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // barrier inits are visible cluster-wide before any remote access (waited below)
  const uint32_t tmem = bar->tmem_base;
  volatile int* abort_flag = &bar->abort;
  pdl_wait();  // everything below reads what earlier kernels wrote

  // ---- this cluster's pair (the same for both CTAs): later pairs first, so the
  // pairs with the most keys start earliest
  if (warp == 0) {
    const int ppt = 2 * rpt;
    const int R = a.rows.rows_uniform;
    const int np = (R + ppt - 1) / ppt;
    const int w = blockIdx.x >> 1;
    const int pair = np - 1 - w / a.rows.num_seqs;
    const int s = w % a.rows.num_seqs;
    int have = pair >= 0 ? 1 : 0, past = 0;
    if (have && lane == 0) {
      // This CTA's Q tile does not depend on the lengths: start loading it now.
      mbar_arrive_expect_tx(&bar->q_full, 2 * kQBlock);
      for (int db = 0; db < 2; ++db)
        tma_load_3d(sQ + db * kQBlock, &tm_q, &bar->q_full, db * 64, g * G, s * R + pair * ppt + rank * rpt);
    }
    if (have) {
      past = a.past[s];
      if (past < 0 || past + R > a.max_ctx) {
        if (a.status && lane == 0 && rank == 0) atomicOr(a.status, CP_DEV_BOUNDS);
        have = 0;
      }
    }
    if (lane == 0) {
      bar->s = s;
      bar->t0 = pair * ppt;
      bar->rows = R;
      bar->past = past;
      bar->have = have;
      bar->q_issued = pair >= 0 ? 1 : 0;
    }
  }
  __syncthreads();
  cluster_wait();  // the peer's barriers are initialised
  const int s = bar->s, t0 = bar->t0, rows = bar->rows, past = bar->past;
  if (!bar->have) {
    if (threadIdx.x == 0) {
      take_ticket(a);
      volatile int zero = 0;  // a Q load in flight lands before shared memory is released
      if (bar->q_issued) mbar_wait(&bar->q_full, 0, &zero, nullptr);
    }
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, kTmemCols);
    }
    return;
  }
  const int t_end = min(t0 + 2 * rpt, rows);
  const TilePlan plan(past, rows, t_end);
  const int nvt = plan.count;
  const int row0 = s * rows;
  const bool fused = a.fused != 0;

  if (warp < 4) {
  // Each role keeps to its own branch up to the final cluster barrier, so the
  // compiler holds each branch to its own register budget.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPRegsControl));
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      const int plane = s * a.hkv + g;  // (the Q tile was issued right after the dependency wait)
      int issued = -1;
      for (int j = 0; j < nvt; ++j) {
        const int st = j % kPStages;
        if (j >= kPStages && !mbar_wait(&bar->kv_empty[st], ((j / kPStages) - 1) & 1, abort_flag, a.status)) break;
        int tile;
        bool is_new;
        plan.at(j, tile, is_new);
        const int j0 = tile * 128;
        uint8_t* dk = sStage + st * kStageBytes;
        uint64_t* fb = &bar->kv_full[st];
        mbar_arrive_expect_tx(fb, kStageBytes);
        if (is_new && fused) {
          const int rel = j0 - past;  // row of k_new holding key j0 (negative rows read as zero)
          for (int db = 0; db < 2; ++db) tma_load_4d(dk + db * kKHalfBlock, &tm_knh, fb, db * 64, g, rel + rank * 64, s);
          tma_load_4d(dk + kVOff, &tm_vnh, fb, rank * 64, g, rel, s);
        } else {
          for (int db = 0; db < 2; ++db) tma_load_3d(dk + db * kKHalfBlock, &tm_kh, fb, db * 64, j0 + rank * 64, plane);
          tma_load_3d(dk + kVOff, &tm_vh, fb, rank * 64, j0, plane);
        }
        issued = j;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's shared memory is released.
        volatile int zero = 0;
        mbar_wait(&bar->q_full, 0, &zero, nullptr);
        for (int t = max(0, issued - kPStages + 1); t <= issued; ++t)
          mbar_wait(&bar->kv_full[t % kPStages], (t / kPStages) & 1, &zero, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ S issuer (CTA 0)
    // Two threads issue the pair's MMAs: this warp the S = Q K^T of each tile,
    // warp 3 the O += P V.  Each waits only for its own inputs; tcgen05 work of
    // one thread completes in issue order, which is all the commits below rely on.
    // The whole warp runs the loop, converged; one elected lane issues.
    if (rank == 0) {
      const uint64_t q_desc = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc0 = make_sdesc_sw128(smem_u32(sStage), 16, 1024);
      constexpr uint64_t kStageStep = kStageBytes >> 4;
      bool ok = warp_wait_cl(&bar->q_ready, 0, abort_flag, a.status);
      for (int j = 0; ok && j < nvt; ++j) {
        // S buffer j % 2 is free once both CTAs read out S of tile j-2.
        if (j >= kSBufs && !warp_wait_cl(&bar->s_free[j % kSBufs], ((j - kSBufs) / kSBufs) & 1, abort_flag, a.status))
          break;
        if (!warp_wait_cl(&bar->kv_ready[j % kPStages], (j / kPStages) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint64_t kd = k_desc0 + (uint64_t)(j % kPStages) * kStageStep;
        const uint32_t d = tmem + 128u * (uint32_t)(j % kSBufs);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oq = ((kk >> 2) * kQBlock + (kk & 3) * 32) >> 4;
          const uint64_t ok2 = ((kk >> 2) * kKHalfBlock + (kk & 3) * 32) >> 4;
          mma_ss_pair_elect(d, q_desc + oq, kd + ok2, kIdescQK, kk > 0);
        }
        mma_commit_pair_elect(&bar->s_full[j % kSBufs], 0x3);
      }
      // Every S MMA issued completes before shared memory or TMEM is released
      // (wait even after an abort).
      mma_commit_pair_elect(&bar->qk_final, 0x1);
      volatile int zero = 0;
      mbar_wait(&bar->qk_final, 0, &zero, a.status);
      __syncwarp();
    }
  } else if (warp == 2) {
    // ================================================================ forwarder
    // Every CTA has read its length (before the __syncthreads above); the last
    // one to take a ticket advances them all.  The atomic's latency overlaps the
    // wait for the Q tile.
    if (lane == 0) take_ticket(a);
    bool ok = warp_wait(&bar->q_full, 0, abort_flag, a.status);
    if (ok && lane == 0) arrive_leader(&bar->q_ready, rank);
    uint8_t* vbase = sStage + kVOff;
    for (int j = 0; ok && j < nvt; ++j) {
      const int st = j % kPStages;
      if (!warp_wait(&bar->kv_full[st], (j / kPStages) & 1, abort_flag, a.status)) break;
      int tile, lo, hi;
      bool is_new;
      plan.at(j, tile, is_new);
      plan.range(tile, is_new, lo, hi);
      if (!(is_new && fused)) {
        // Read from the cache: V rows at or past `hi` hold no key of this walk
        // (unwritten or stale slots, possibly being written by this launch's append).
        const int z0 = max(hi - tile * 128, 0);
        if (z0 < 128) {
          uint4* p = reinterpret_cast<uint4*>(vbase + st * kStageBytes + z0 * 128);
          for (int e = lane; e < (128 - z0) * 8; e += 32) p[e] = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) arrive_leader(&bar->kv_ready[st], rank);
    }
  } else if (warp == 3) {
    // ================================================================ fused append
    // The K/V rows of this Q tile's tokens for KV head g go to their slots
    // past + t of the cache ([Wiki] 一.1); every (token, KV head) row of the
    // chunk belongs to exactly one Q tile.  Read-only for the attention: the
    // tiles that hold these keys are read from k_new / v_new.
    if (fused) {
      const int tk0 = t0 + rank * rpt, tk1 = min(tk0 + rpt, rows);
      const int nrow = max(tk1 - tk0, 0);
      const long long src_row = (long long)row0 + tk0;  // token row of k_new
      const long long dst_row = ((long long)(s * a.hkv + g)) * a.capacity + past + tk0;
      for (int e = lane; e < nrow * 16; e += 32) {
        const int r = e >> 4, c = e & 15;  // 16 vectors of 16 bytes per 128-element row
        const long long so = ((src_row + r) * a.hkv + g) * 16 + c;
        const long long dof = (dst_row + r) * 16 + c;
        const uint4 kv = reinterpret_cast<const uint4*>(a.k_new)[so];
        const uint4 vv = reinterpret_cast<const uint4*>(a.v_new)[so];
        reinterpret_cast<uint4*>(a.k_cache)[dof] = kv;
        reinterpret_cast<uint4*>(a.v_cache)[dof] = vv;
      }
    }
    if (rank == 0) {
      // ================================================================ P V issuer (CTA 0)
      const uint64_t v_desc0 = make_sdesc_sw128(smem_u32(sStage + kVOff), kQBlock, 1024);
      constexpr uint64_t kStageStep = kStageBytes >> 4;
      for (int i = 0; i < nvt; ++i) {
        if (!warp_wait_cl(&bar->p_ready[i % kSBufs], (i / kSBufs) & 1, abort_flag, a.status)) break;
        // The tile's V halves landed before its S was computed (same stage).
        tc_fence_after();
        const uint64_t vd = v_desc0 + (uint64_t)(i % kPStages) * kStageStep;
        const uint32_t p = tmem + kColP + 64u * (uint32_t)(i % kSBufs);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)
          mma_ts_pair_elect(tmem + kColO, p + kk * 8, vd + ((kk * 2048) >> 4), kIdescPV,
                            (i > 0 || kk > 0) ? 1u : 0u);
        // The stage's K (read by S of this tile, complete before its P existed)
        // and V are free; P V of this tile is done.
        mma_commit_pair_elect(&bar->kv_empty[i % kPStages], 0x3);
        mma_commit_pair_elect(&bar->o_done[i % kORing], 0x3);
      }
      // Every P V issued (they write both CTAs' TMEM and read both CTAs' shared
      // memory) completes before either CTA releases them; wait even after an abort.
      mma_commit_pair_elect(&bar->o_final, 0x3);
      volatile int zero = 0;
      mbar_wait(&bar->o_final, 0, &zero, a.status);
      __syncwarp();
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPRegsSoftmax));
    // ================================================================ softmax warps
    // Warpgroup wg takes the tiles i with i % 2 == wg; thread (warp, lane) owns
    // row 32 * (warp % 4) + lane and all 128 keys of each of its tiles.
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;              // TMEM lanes [32*quarter, +32)
    const int m = quarter * 32 + lane;         // this thread's row of the CTA's Q tile
    const int tok = t0 + rank * rpt + m / G;
    const int head = g * G + m % G;
    const bool row_ok = tok < t_end;
    const int p_row = row_ok ? past + tok : -1;  // absolute query position
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = a.scale_log2;
    // Named barriers handing the running max between the two warps of a row
    // (warp quarter+4 and quarter+8): tiles of warpgroup 0 -> 1 use ids 1-4,
    // 1 -> 0 ids 5-8.  Each is a producer arrive / consumer sync pair made in
    // every iteration whatever happens, so no warp can be left waiting.
    const int id_send = 1 + quarter + 4 * wg, id_recv = 1 + quarter + 4 * (wg ^ 1);
    // P-ready and S-free: every softmax warp arrives on CTA 0's barriers itself
    // (CTA 1's warps with a remote arrive).
    float m_used = -INFINITY;  // max (log2 domain) this warpgroup last exponentiated against
    float l_part = 0.f;        // this warpgroup's share of the row sum, relative to m_used
    bool good = true;
    for (int i = wg; i < nvt; i += 2) {
      const int b = i % kSBufs;
      const bool got = warp_wait(&bar->s_full[b], (i / kSBufs) & 1, abort_flag, a.status);
      tc_fence_after();
      good = good && got;
      uint32_t sv[128];
      const uint32_t s_col = tmem + lane_off + 128u * (uint32_t)b;
      if (good) {
        tmem_ld32(s_col + 0, &sv[0]);
        tmem_ld32(s_col + 32, &sv[32]);
        tmem_ld32(s_col + 64, &sv[64]);
        tmem_ld32(s_col + 96, &sv[96]);
        tmem_wait_ld();
        // S buffer b may take the scores of tile i+2.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader_light(&bar->s_free[b], rank);
      }
      int tile, lo, hi;
      bool is_new;
      plan.at(i, tile, is_new);
      plan.range(tile, is_new, lo, hi);
      // Visible columns: [c_lo, c_hi) (keys of this walk, at or before the row).
      const int k0 = tile * 128;
      const int c_lo = lo - k0, c_hi = min(hi, p_row + 1) - k0;
      if (c_lo > 0 || c_hi < 128) {  // not fully visible: mask first
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < c_lo || c >= c_hi) sv[c] = __float_as_uint(-INFINITY);
      }
      float mx;
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
      // The running max after tile i-1, from the other warpgroup.
      float m_prev = -INFINITY;
      if (i > 0) {
        bar_named(id_recv, 64);
        m_prev = bar->xmax[wg ^ 1][0][m];
      }
      // The max is raised only when it grows by more than 2^kRescaleLog2 (a
      // row-local decision), so most tiles need no rescale of O.
      const bool grow = mx2 > m_prev + kRescaleLog2 || (m_prev == -INFINITY && mx2 != -INFINITY);
      const float m_i = grow ? mx2 : m_prev;
      if (i + 1 < nvt) {
        bar->xmax[wg][0][m] = m_i;
        bar_arrive(id_send, 64);
      }
      const float neg_m = (m_i == -INFINITY) ? 0.f : -m_i;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float x0 = __uint_as_float(sv[2 * c]), x1 = __uint_as_float(sv[2 * c + 1]);
        ffma2(x0, x1, sl2, neg_m);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        fadd2(ps4[2 * (c & 1)], ps4[2 * (c & 1) + 1], p0, p1);
        sv[c] = pack2<T>(p0, p1);  // P (16-bit pairs) overwrites the front of sv
      }
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      l_part = (m_used == -INFINITY ? 0.f : l_part * ex2_approx(m_used - m_i)) + psum;
      m_used = m_i;
      if (i > 0 && __any_sync(0xffffffffu, grow && m_prev != -INFINITY)) {
        // Rows whose max grew rescale O (P V of tiles < i, relative to m_prev)
        // once P V of tile i-1 has completed (P V runs in issue order).  Slot
        // (i-1) % 8 of the o_done ring last held P V of tile i-9, completed
        // before P V of tile i-4, which this warpgroup saw complete at its
        // previous tile; P V of tile i+7 is far from issued.  So the parity of
        // phase (i-1) / 8 tells whether P V of tile i-1 is done.  sv[64..95] (S
        // values already used) stage O.
        const float alpha = (grow && m_prev != -INFINITY) ? ex2_approx(m_prev - m_i) : 1.f;
        if (!warp_wait(&bar->o_done[(i - 1) % kORing], ((i - 1) / kORing) & 1, abort_flag, a.status)) good = false;
        tc_fence_after();
        if (good) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t o_col = tmem + lane_off + kColO + 32u * (uint32_t)c;
            tmem_ld32(o_col, &sv[64]);
            tmem_wait_ld();
#pragma unroll
            for (int e = 64; e < 96; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * alpha);
            tmem_st32(o_col, &sv[64]);
            tmem_wait_st();
          }
        }
      }
      if (good && i >= kSBufs) {
        // P buffer b is free once P V of tile i-2 has completed.  Slot
        // (i-2) % 8 of the o_done ring last held P V of tile i-10, completed
        // before P V of tile i-4, which this warpgroup saw complete at its
        // previous tile (every warpgroup waits here at each of its tiles).
        if (!warp_wait(&bar->o_done[(i - 2) % kORing], ((i - 2) / kORing) & 1, abort_flag, a.status)) good = false;
        tc_fence_after();
      }
      if (good) {
        const uint32_t p_col = tmem + lane_off + kColP + 64u * (uint32_t)b;
        tmem_st32(p_col, &sv[0]);
        tmem_st32(p_col + 32, &sv[32]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader_light(&bar->p_ready[b], rank);
      }
    }

    // ================================================================ epilogue
    // O is relative to the max after the last tile; each warpgroup's share of the
    // row sum is relative to the max it last used.  Warpgroup wg finishes head
    // dims [64 wg, 64 wg + 64) of every row.
    bool fin = good;
    if (fin) fin = warp_wait(&bar->o_final, 0, abort_flag, a.status);
    tc_fence_after();
    bar->xmax[wg][1][m] = m_used;
    bar->xsum[wg][m] = l_part;
    fin = bar_and(9, 256, fin);
    const int half = wg;
    const int tile_tok0 = t0 + rank * rpt;
    const bool full_tile = tile_tok0 + rpt <= t_end;
    const bool own_rows = tile_tok0 < t_end;
    if (fin && own_rows) {
      const float ma = bar->xmax[0][1][m], mb = bar->xmax[1][1][m];
      const float mf = fmaxf(ma, mb);
      const float la = ma == -INFINITY ? 0.f : bar->xsum[0][m] * ex2_approx(ma - mf);
      const float lb = mb == -INFINITY ? 0.f : bar->xsum[1][m] * ex2_approx(mb - mf);
      const float lsum = la + lb;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const uint32_t o_col = tmem + lane_off + kColO + 64u * (uint32_t)half;
      uint8_t* box = sQ + half * kQBlock + m * 128;  // this half's 64 dims of row m (128B-swizzled)
      T* out = static_cast<T*>(a.out) + ((long long)(row0 + tok) * a.hq + head) * D + 64 * half;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_col + 32 * c, ov);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<T>(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
        if (full_tile) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int chunk = c * 4 + e;
            *reinterpret_cast<uint4*>(box + ((chunk ^ (m & 7)) * 16)) =
                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
    if (full_tile) {
      fence_proxy_async_smem();  // the TMA store reads the tile through the async proxy
      bar_named(10, 256);
      if (warp == 4 && lane == 0 && fin) {
        for (int db = 0; db < 2; ++db) tma_store_3d(&tm_o, sQ + db * kQBlock, db * 64, g * G, row0 + tile_tok0);
        bulk_commit_group();
        bulk_wait_read_all();  // the staging buffer is read out; the writes finish with the grid
      }
    }
  }

  // Both CTAs leave together: every MMA has completed (CTA 0's issuer waited)
  // and every remote arrive has landed before shared memory or TMEM is released.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <typename T>
cudaError_t launch_t(const PairArgs& a, const CUtensorMap& tq, const CUtensorMap& to, const CUtensorMap& tkh,
                     const CUtensorMap& tvh, const CUtensorMap& tknh, const CUtensorMap& tvnh, int pairs_bound,
                     cudaStream_t st) {
  const uint32_t smem = PairSmem::alloc;
  static std::atomic<uint64_t> ready_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready_mask.load(std::memory_order_acquire) & bit)) {
    // The register split is only sound at the per-thread count it was sized
    // for: refuse to launch a build that came out at another count.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_pair_kernel<T>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kPRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(attn_pair_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ready_mask.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * pairs_bound, a.hkv);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, attn_pair_kernel<T>, tq, to, tkh, tvh, tknh, tvnh, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool attn_pair_supported(int d, int group, int dtype) {
  return d == 128 && group >= 1 && group <= 16 && (group & (group - 1)) == 0 && (dtype == CP_BF16 || dtype == CP_F16);
}

cudaError_t launch_attn_pair(const PairArgs& a, int dtype, const CUtensorMap& tq, const CUtensorMap& to,
                             const CUtensorMap& tkh, const CUtensorMap& tvh, const CUtensorMap& tknh,
                             const CUtensorMap& tvnh, int pairs_bound, cudaStream_t st) {
  if (pairs_bound <= 0) return cudaSuccess;
  if (dtype == CP_BF16) return launch_t<__nv_bfloat16>(a, tq, to, tkh, tvh, tknh, tvnh, pairs_bound, st);
  return launch_t<__half>(a, tq, to, tkh, tvh, tknh, tvnh, pairs_bound, st);
}

}  // namespace cp
