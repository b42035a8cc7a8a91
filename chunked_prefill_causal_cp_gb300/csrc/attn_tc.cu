// attn_tc.cu -- chunk attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ([Wiki] 一.2; [Glossary] "How chunked prefill works"): row i
// of a chunk is the query at absolute position p = past + i and attends to
// the keys at positions [0, p] -- the cached prefix plus its own causal
// triangle -- over a cache at fixed physical capacity, a paged pool, or a
// right-aligned rolling window ([Horizon] 3-4).
//
// Tiling.  One CTA computes one 128-row M tile.  GroupQueryAttention packs the
// G = Hq/Hkv query heads of one KV head into the tile: 128/G consecutive
// tokens x G heads, row m <-> (token m / G, head m % G), so every K/V tile
// loaded into shared memory serves all heads of the group.  K/V tiles hold
// 128 keys and start at absolute key 0, so tile boundaries never depend on
// the chunk's width (padded and unpadded runs see the same tiles); tiles past
// the tile's last query position are never loaded (causal tile skip).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K and V tiles into a 2-stage ring.
//   warp 1      TMEM allocator and MMA issuer (one elected lane):
//               S = Q K^T  (A = Q, B = K, both K-major, from shared memory),
//               O += P V   (A = P from TMEM, B = V MN-major from shared memory).
//   warps 2-5   softmax: thread m owns row m (TMEM lane m).  It reads the
//               S row from TMEM, masks by absolute position, keeps the running
//               max / sum in the log2 domain, writes P (16-bit) over the S
//               columns it came from, rescales its O row in TMEM when the max
//               grows, and finally normalises O and stores it.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+D).  Two S
// buffers let the tensor core compute S_{j+1} while softmax works on S_j.
//
// Shared memory (128-byte swizzle, what TMA writes and the MMA descriptors
// read): Q [D/64][128 rows][128 B]; K and V [2 stages][D/64][128 rows][128 B].
//
// Keys beyond the written length inside the last tile may hold stale or
// poisoned bytes; their scores are masked and the MMA warp zeroes those V rows
// before P V, so 0 * garbage never reaches O.
#include <cmath>
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kBlockBytes = 128 * 128;  // [128 rows][64 x 16-bit] = 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;

struct __align__(8) TcBarriers {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_ready[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct TcSmem {
  static constexpr int DB = D / 64;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + DB * kBlockBytes;
  static constexpr uint32_t v_off = k_off + kStages * DB * kBlockBytes;
  static constexpr uint32_t bar_off = v_off + kStages * DB * kBlockBytes;
  static constexpr uint32_t bytes = bar_off + sizeof(TcBarriers);
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

// Which (sequence, first token) this CTA owns.  Within a sequence the tiles are
// handed out last-first, so the tiles with the most keys start earliest.
__device__ __forceinline__ bool find_tile(const AttnArgs& a, int rpt, int w, int& s, int& t0) {
  if (a.rows.rows_uniform > 0) {
    const int nt = (a.rows.rows_uniform + rpt - 1) / rpt;
    const int tile = nt - 1 - w / a.rows.num_seqs;
    s = w % a.rows.num_seqs;
    if (tile < 0) return false;
    t0 = tile * rpt;
    return true;
  }
  for (int q = 0; q < a.rows.num_seqs; ++q) {
    const int r = seq_rows(a.rows, q);
    if (r < a.min_rows) continue;
    const int nt = (r + rpt - 1) / rpt;
    if (w < nt) {
      s = q;
      t0 = (nt - 1 - w) * rpt;
      return true;
    }
    w -= nt;
  }
  return false;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int rpt = kTcBlockM / G;
  const int g = blockIdx.y;

  // ---- this CTA's tile (uniform across the CTA; exits before any setup)
  int s, t0;
  if (!find_tile(a, rpt, blockIdx.x, s, t0)) return;
  const int rows = seq_rows(a.rows, s);
  const int past = a.past[s];
  const int n = past + rows;  // positions written, including this call's rows
  if (past < 0 || n > a.max_ctx) {
    if (a.status && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int row0 = seq_row0(a.rows, s);
  const int t_end = min(t0 + rpt, rows);
  const bool rolling = a.cache.kind == CP_CACHE_ROLLING;
  const int cap = a.cache.capacity;
  // Key indices walked: absolute positions [0, nkeys) (contiguous / paged) or
  // physical ring slots [0, nkeys) (rolling).
  const int nkeys = rolling ? min(n, cap) : past + t_end;
  const int n_valid = rolling ? nkeys : n;  // key indices holding written data
  const int ntiles = (nkeys + kTcBlockN - 1) / kTcBlockN;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar->k_full[i], 1);
      mbar_init(&bar->k_empty[i], 1);
      mbar_init(&bar->v_full[i], 1);
      mbar_init(&bar->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_ready[i], 128);
    }
    mbar_init(&bar->o_done, 1);
    mbar_init(&bar->drain, 1);
    bar->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  volatile int* abort_flag = &bar->abort;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bar->q_full, DB * kBlockBytes);
      for (int db = 0; db < DB; ++db)
        tma_load_3d(sQ + db * kBlockBytes, &tm_q, &bar->q_full, db * 64, g * G, row0 + t0);
      const int ps = a.cache.page_size;
      int last_issued = -1;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        const int j0 = j * kTcBlockN;
        for (int which = 0; which < 2; ++which) {  // 0: K, 1: V
          uint64_t* full = which ? &bar->v_full[st] : &bar->k_full[st];
          uint64_t* empty = which ? &bar->v_empty[st] : &bar->k_empty[st];
          const CUtensorMap* map = which ? &tm_v : &tm_k;
          uint8_t* dst = (which ? sV : sK) + st * DB * kBlockBytes;
          if (!mbar_wait(empty, ph ^ 1, abort_flag, a.status)) break;
          if (a.cache.kind != CP_CACHE_PAGED) {
            mbar_arrive_expect_tx(full, DB * kBlockBytes);
            for (int db = 0; db < DB; ++db)
              tma_load_3d(dst + db * kBlockBytes, map, full, db * 64, j0, s * a.hkv + g);
          } else {
            // One box of `ps` rows per page that holds at least one written key.
            const int npg = kTcBlockN / ps;
            int pages[kTcBlockN / 16];
            int cnt = 0;
            for (int pi = 0; pi < npg; ++pi) {
              const int key = j0 + pi * ps;
              int page = -1;
              if (key < n_valid) {
                const int blk = key / ps;
                if (blk < a.cache.max_blocks) page = a.cache.block_table[(long long)s * a.cache.max_blocks + blk];
                if (page < 0 || page >= a.cache.num_pages) {
                  if (a.status) atomicOr(a.status, CP_DEV_BOUNDS);
                  page = -1;
                }
              }
              pages[pi] = page;
              cnt += page >= 0;
            }
            mbar_arrive_expect_tx(full, (uint32_t)cnt * DB * ps * 128u);
            for (int pi = 0; pi < npg; ++pi) {
              if (pages[pi] < 0) continue;
              for (int db = 0; db < DB; ++db)
                tma_load_3d(dst + db * kBlockBytes + pi * ps * 128, map, full, db * 64, 0,
                            pages[pi] * a.hkv + g);
            }
          }
        }
        if (*abort_flag) break;
        last_issued = j;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's shared memory is released.
        volatile int zero = 0;
        for (int t = last_issued - 1; t <= last_issued; ++t) {
          if (t < 0) continue;
          mbar_wait(&bar->k_full[t & 1], (t >> 1) & 1, &zero, nullptr);
          mbar_wait(&bar->v_full[t & 1], (t >> 1) & 1, &zero, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    bool ok = ntiles > 0 && warp_wait(&bar->q_full, 0, abort_flag, a.status);
    auto issue_qk = [&](int j) -> bool {
      const int st = j & 1;
      if (!warp_wait(&bar->k_full[st], (j >> 1) & 1, abort_flag, a.status)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + (st ? kColS1 : kColS0);
        const uint32_t q_base = smem_u32(sQ);
        const uint32_t k_base = smem_u32(sK + st * DB * kBlockBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          mma_ss(d_tmem, make_sdesc_sw128(q_base + off, 16, 1024), make_sdesc_sw128(k_base + off, 16, 1024),
                 kIdescQK, kk > 0);
        }
        mma_commit(&bar->s_full[st]);
        mma_commit(&bar->k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_qk(0);
    if (ok && ntiles > 1) ok = issue_qk(1);
    for (int j = 0; ok && j < ntiles; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!warp_wait(&bar->p_ready[st], ph, abort_flag, a.status)) break;
      if (!warp_wait(&bar->v_full[st], ph, abort_flag, a.status)) break;
      tc_fence_after();
      uint8_t* v_stage = sV + st * DB * kBlockBytes;
      if (j == ntiles - 1) {
        const int tail = n_valid - j * kTcBlockN;  // rows >= tail hold no written key
        if (tail < kTcBlockN) {
          for (int db = 0; db < DB; ++db) {
            uint4* p = reinterpret_cast<uint4*>(v_stage + db * kBlockBytes + tail * 128);
            const int nvec = (kTcBlockN - tail) * 128 / 16;
            for (int i = lane; i < nvec; i += 32) p[i] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t p_tmem = tmem + (st ? kColS1 : kColS0);
        const uint32_t v_base = smem_u32(v_stage);
#pragma unroll
        for (int kk = 0; kk < kTcBlockN / 16; ++kk)
          mma_ts(tmem + kColO, p_tmem + kk * 8, make_sdesc_sw128(v_base + kk * 2048, kBlockBytes, 1024),
                 kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar->o_done);
        mma_commit(&bar->v_empty[st]);
      }
      __syncwarp();
      if (j + 2 < ntiles) ok = issue_qk(j + 2);
    }
    // Make sure every MMA this warp issued has finished before TMEM is freed.
    if (lane == 0 && ntiles > 0) mma_commit(&bar->drain);
    __syncwarp();
    if (ntiles > 0) {
      volatile int zero = 0;  // wait even after an abort: MMAs may still be in flight
      warp_wait(&bar->drain, 0, &zero, a.status);
    }
  } else {
    // ================================================================ softmax
    const int quarter = warp & 3;            // TMEM lanes [32*quarter, +32)
    const int mrow = quarter * 32 + lane;    // this thread's row of the tile
    const int tok = t0 + mrow / G;
    const int head = g * G + mrow % G;
    const bool row_ok = tok < t_end;
    const int p_row = row_ok ? past + tok : -1;  // absolute query position
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int lo = rolling ? max(a.left_pad ? a.left_pad[s] : 0, 0) : 0;
    // Rolling: slot -> absolute position (see cp_kv.cuh), split at slot r.
    const int r_slot = n > 0 ? (n - 1) % cap : 0;
    const int base_hi = n - 1 - r_slot;
    const float sl2 = a.scale_log2;

    float m_run = -INFINITY, l_run = 0.f;
    bool alive = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (!warp_wait(&bar->s_full[st], (j >> 1) & 1, abort_flag, a.status)) { alive = false; break; }
      tc_fence_after();
      const uint32_t s_col = lane_base + (st ? kColS1 : kColS0);
      uint32_t sv[128];
      tmem_ld32(s_col + 0, &sv[0]);
      tmem_ld32(s_col + 32, &sv[32]);
      tmem_ld32(s_col + 64, &sv[64]);
      tmem_ld32(s_col + 96, &sv[96]);
      tmem_wait_ld();
      const int j0 = j * kTcBlockN;
      float mx = -INFINITY;
      if (!rolling && j0 + kTcBlockN - 1 <= p_row) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float x = __uint_as_float(sv[c]) * sl2;
          sv[c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = j0 + c;
          bool vis;
          if (!rolling) {
            vis = key <= p_row;
          } else {
            const int pos = key + base_hi - (key > r_slot ? cap : 0);
            vis = key < nkeys && pos >= lo && pos <= p_row;
          }
          const float x = vis ? __uint_as_float(sv[c]) * sl2 : -INFINITY;
          sv[c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_run == -INFINITY) ? (m_new == -INFINITY ? 1.f : 0.f) : ex2_approx(m_run - m_new);
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2_approx(__uint_as_float(sv[2 * c]) - m_use);
        const float p1 = ex2_approx(__uint_as_float(sv[2 * c + 1]) - m_use);
        psum += p0 + p1;
        sv[c] = pack2<T>(p0, p1);
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      tmem_st32(s_col + 0, &sv[0]);
      tmem_st32(s_col + 32, &sv[32]);
      tmem_wait_st();
      if (j > 0) {
        // O holds P V of tiles < j; rescale it before P_j V_j is added.
        if (!warp_wait(&bar->o_done, (j - 1) & 1, abort_flag, a.status)) { alive = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(lane_base + kColO + 32 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(lane_base + kColO + 32 * c, ov);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(&bar->p_ready[st]);
    }
    // ---- epilogue: O / l -> out
    if (alive && ntiles > 0 && warp_wait(&bar->o_done, (ntiles - 1) & 1, abort_flag, a.status)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      T* out = static_cast<T*>(a.out) + ((long long)(row0 + tok) * a.hq + head) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + 32 * c, ov);
        tmem_wait_ld();
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2<T>(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    } else if (ntiles == 0 && row_ok) {
      // No key visible at all (e.g. a rolling left-pad query): output 0.
      T* out = static_cast<T*>(a.out) + ((long long)(row0 + tok) * a.hq + head) * D;
      for (int e = 0; e < D; ++e) out[e] = T(0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D>
cudaError_t launch_t(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     int tiles_bound, cudaStream_t st) {
  // D = 64 would fit two CTAs per SM, but each CTA takes all 512 TMEM
  // columns; ask for enough shared memory to keep it at one CTA per SM.
  const uint32_t smem = TcSmem<D>::alloc < 120u * 1024u ? 120u * 1024u : TcSmem<D>::alloc;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(tiles_bound, a.hkv);
  attn_tc_kernel<T, D><<<grid, kThreads, smem, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(int d, int group, int dtype) {
  return (d == 64 || d == 128) && group >= 1 && group <= 16 && (group & (group - 1)) == 0 &&
         (dtype == CP_BF16 || dtype == CP_F16);
}

cudaError_t launch_attn_tc(const AttnArgs& a, int dtype, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, int tiles_bound, cudaStream_t st) {
  if (tiles_bound <= 0) return cudaSuccess;
  if (dtype == CP_BF16)
    return a.d == 64 ? launch_t<__nv_bfloat16, 64>(a, tq, tk, tv, tiles_bound, st)
                     : launch_t<__nv_bfloat16, 128>(a, tq, tk, tv, tiles_bound, st);
  return a.d == 64 ? launch_t<__half, 64>(a, tq, tk, tv, tiles_bound, st)
                   : launch_t<__half, 128>(a, tq, tk, tv, tiles_bound, st);
}

}  // namespace cp
