// decode.cu -- single-row (decode) attention on the memory-bound split-KV path.
//
// A decode row reads its sequence's whole K/V once and does ~1 FLOP per byte
// (Ultralytics glossary "Chunked Prefill", "Prefill, decode and generation
// stalls": decode is memory-bandwidth bound), so this path is built around
// coalesced 16-byte loads, not the tensor cores.
//
// decode_split_kernel: one CTA per (split of 512 keys, KV head, sequence).
//   The GQA group's query heads share every K/V row the CTA loads.  A group
//   of D/16 lanes holds one key row (16 elements = two 16-byte loads per
//   lane); each lane keeps the group's q values for its 16 dimensions, the
//   products accumulate with packed fp32x2 FMAs, the partial dot products
//   are reduced with xor shuffles, scores go to shared memory, the CTA takes
//   the split's max and sum (log2 domain), then streams V once (again with
//   packed FMAs) and writes the unnormalised partial output.  Instruction
//   count per loaded byte, not bandwidth, is what limits this path, hence
//   the wide lanes and packed arithmetic.
// decode_combine_kernel: merges a row's split partials in split order
//   (log-sum-exp), so the result depends only on the row's own context.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kDecConsumers = 4;     // consumer warps per CTA (plus an issuer and a resolver warp)
constexpr int kDecCtasPerSm = 3;     // resident CTAs per SM of the persistent grid
constexpr int kDecStageBytes = 8192; // one ring stage: 32 rows at D = 128, 64 at D = 64
constexpr int kDecStages = 5;        // ring depth
constexpr int kDecSlots = 3;         // resolved items held ahead of the consumers

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

// Two 16-bit values packed in a 32-bit word -> (low, high) as floats.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// (a.x, a.y) += (b.x, b.y) * (c.x, c.y) as one packed instruction.
__device__ __forceinline__ void ffma2v(float2& a, float2 b, float2 c) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\tmov.b64 rc, {%4, %5};\n\t"
      "fma.rn.f32x2 ra, rb, rc, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a.x), "+f"(a.y)
      : "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
}

// Shared-memory plan of decode_split_kernel<T, D, H>.
template <int D, int H>
struct DecSmem {
  static constexpr int kRow = D * 2;                        // bytes of one K or V row
  static constexpr int kStageRows = kDecStageBytes / kRow;  // 32 (D = 128) or 64 (D = 64)
  static constexpr int ring = 0;                                      // [kDecStages][kDecStageBytes]
  static constexpr int q = ring + kDecStages * kDecStageBytes;        // 16-bit [kDecSlots][H][D]
  static constexpr int rows = q + kDecSlots * H * D * 2;              // uint32 [kDecSlots][kDecodeSplit]
  static constexpr int pages = rows + kDecSlots * 4 * kDecodeSplit;   // int [kDecodeSplit + 1] (resolver)
  static constexpr int sc = pages + 4 * (kDecodeSplit + 4);           // float [H][kDecodeSplit]
  static constexpr int red = sc + 4 * H * kDecodeSplit;               // float [kDecConsumers][H][D]
  static constexpr int bars = red + 4 * kDecConsumers * H * D;        // uint64 full, empty, ready, freed
  static constexpr int items = bars + 8 * (2 * kDecStages + 2 * kDecSlots);  // int [kDecSlots][2]
  static constexpr int misc = items + 8 * kDecSlots;                  // int bad[kDecSlots], abort
  static constexpr int ml = misc + 4 * (kDecSlots + 1);               // float max[kDecConsumers][H], sum[..][H]
  static constexpr int bytes = ml + 8 * kDecConsumers * H;
  static_assert(kDecCtasPerSm * (bytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

// Row index (in rows of D elements) of an invalid key: never copied.
constexpr uint32_t kNoRow = 0xffffffffu;

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDecConsumers * 32) : "memory"); }

// Named barrier over the consumer warps that also ORs a predicate across them.
__device__ __forceinline__ bool consumers_sync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kDecConsumers * 32)
      : "memory");
  return r != 0;
}

// Row of a staged tile, as the two 16-byte chunks c0 = sub and c1 = sub + LPK.
__device__ __forceinline__ void lds_row(const unsigned char* row, int sub, int lpk, uint32_t (&w)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(row + sub * 16);
  const uint4 b = *reinterpret_cast<const uint4*>(row + (sub + lpk) * 16);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// A work item: one split of kDecodeSplit keys, for H query heads of one KV
// group of one decode sequence.  Ids run sequence-major, then split, then
// head block, so the H-head blocks of one split are neighbours (a group of 8
// heads takes two blocks that read the same rows close together in time, the
// second mostly from L2), and a sequence's empty splits (those past its
// length) are the tail of its id range, which a claim skips in one step.
struct DecItem {
  int s, split, hb, nk;
};

__device__ __forceinline__ void dec_ids(const AttnArgs& a, int id, int nhb, DecItem& it) {
  it.hb = id % nhb;
  it.split = (id / nhb) % a.max_splits;
  it.s = (id / nhb) / a.max_splits;
}

__device__ __forceinline__ bool dec_item(const AttnArgs& a, int id, int nhb, DecItem& it) {
  dec_ids(a, id, nhb, it);
  if (seq_rows(a.rows, it.s) != 1) return false;
  const int past = a.past[it.s];
  const int n = past + 1;
  if (past < 0 || n > a.max_ctx) {
    if (a.status && it.split == 0 && it.hb == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return false;
  }
  const int k0 = it.split * kDecodeSplit;
  if (k0 >= n) return false;
  it.nk = min(n - k0, kDecodeSplit);
  return true;
}

// Persistent split-KV decode: kDecCtasPerSm CTAs per SM, each with
// kDecConsumers consumer warps, an issuer warp and a resolver warp.
//
// The resolver claims work items from a device counter (lane 0, one atomic
// per claim, the next claim issued ahead; a claim that lands on a sequence's
// empty tail moves the counter to the next sequence), reads the sequence's
// length and page table, and writes the item's row indices into one of
// kDecSlots item slots, up to kDecSlots items ahead of the consumers, so the
// latency of those reads is off the copy path.  The issuer streams each
// resolved item's q heads, then its K rows, then its V rows through a ring of
// kDecStages stages with bulk copies: one copy per run of contiguous rows (a
// whole stage for a contiguous cache, one page per copy for a paged one).  It
// runs across item boundaries without a gap, so the ring stays full and the
// bytes in flight are bounded by shared memory, not registers.  After the last
// item both pass a sentinel that ends the consumers.
//
// In the K phase the consumers take a row per group of LPK = D/16 lanes, 16
// elements per lane (chunks sub and sub + LPK, so a quarter-warp reads 128
// contiguous bytes), with packed fp32x2 FMAs; scores go to shared memory, the
// split's max and sum are taken in the log2 domain, the V stages are
// accumulated with D/8 lanes per row (half the accumulator registers),
// warps' partial sums are added in a fixed order and the unnormalised partial
// output is written for the combine kernel.
template <typename T, int D, int H>
__global__ void __launch_bounds__((kDecConsumers + 2) * 32, kDecCtasPerSm)
    decode_split_kernel(const AttnArgs a, int* counter) {
  using L = DecSmem<D, H>;
  constexpr int LPK = D / 16;               // lanes per row (K phase)
  constexpr int KPW = 32 / LPK;             // rows per warp per stage
  constexpr int SR = L::kStageRows;
  constexpr int NST = kDecStages;
  constexpr int NSL = kDecSlots;
  constexpr int KPP = kDecConsumers * KPW;  // rows per K pass of all consumers
  constexpr int KPASS = SR / KPP;
  static_assert(KPASS * KPP == SR, "K passes cover a stage");
  static_assert(SR % 32 == 0, "the issuer covers a stage in rounds of 32 rows");
  constexpr int LPV = D / 8;                // lanes per row in the V phase
  constexpr int RPW = 32 / LPV;             // rows per warp per V pass
  constexpr int VPASS = SR / (kDecConsumers * RPW);
  static_assert(VPASS * kDecConsumers * RPW == SR, "V passes cover a stage");
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty = full + NST;
  uint64_t* ready = empty + NST;
  uint64_t* freed = ready + NSL;
  int* s_items = reinterpret_cast<int*>(smem + L::items);
  int* s_bad = reinterpret_cast<int*>(smem + L::misc);
  volatile int* s_abort = s_bad + NSL;
  float (*s_wmax)[H] = reinterpret_cast<float (*)[H]>(smem + L::ml);            // per warp, per head
  float (*s_psum)[H] = reinterpret_cast<float (*)[H]>(smem + L::ml + 4 * kDecConsumers * H);

  pdl_launch_dependents();
  const int nhb = a.hq / H;
  const int total = a.max_splits * a.rows.num_seqs * nhb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecConsumers);
    }
    for (int i = 0; i < NSL; ++i) {
      mbar_init(&ready[i], 1);
      mbar_init(&freed[i], kDecConsumers);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // everything below reads what earlier kernels wrote

  if (warp == kDecConsumers + 1) {
    // ------------------------------------------------ resolver warp
    int* s_pg = reinterpret_cast<int*>(smem + L::pages);
    int next = lane == 0 ? atomicAdd(counter, 1) : 0;
    for (int j = 0;; ++j) {
      const int sl = j % NSL;
      DecItem it;
      int id;
      for (;;) {
        id = __shfl_sync(0xffffffffu, next, 0);
        if (id >= total) break;
        if (lane == 0) next = atomicAdd(counter, 1);
        if (dec_item(a, id, nhb, it)) break;
        // Every later id of this sequence is empty too: move the counter past them.
        if (lane == 0) atomicMax(counter, (it.s + 1) * a.max_splits * nhb);
      }
      if (j >= NSL && !warp_wait(&freed[sl], ((j - NSL) / NSL) & 1, s_abort, a.status)) return;
      if (id >= total) {  // sentinel
        if (lane == 0) {
          s_items[sl * 2] = -1;
          mbar_arrive(&ready[sl]);
        }
        return;
      }
      const int g = (it.hb * H) / a.group, k0 = it.split * kDecodeSplit;
      uint32_t* rows = reinterpret_cast<uint32_t*>(smem + L::rows) + sl * kDecodeSplit;
      bool bad = false;
      if (a.cache.kind == CP_CACHE_PAGED) {
        // The item's page ids first (one load per page, all in flight together),
        // then each row from its page.
        const int ps = a.cache.page_size;
        const int b0 = k0 / ps, nb = (k0 + it.nk - 1) / ps - b0 + 1;
        for (int b = lane; b < nb; b += 32) {
          const int blk = b0 + b;
          int pg = -1;
          if (blk < a.cache.max_blocks) pg = a.cache.block_table[(long long)it.s * a.cache.max_blocks + blk];
          s_pg[b] = (pg >= 0 && pg < a.cache.num_pages) ? pg : -1;
        }
        __syncwarp();
        for (int kk = lane; kk < it.nk; kk += 32) {
          const int jj = k0 + kk;
          const int pg = s_pg[jj / ps - b0];
          rows[kk] = pg < 0 ? kNoRow : (uint32_t)(((long long)pg * a.hkv + g) * ps + jj % ps);
          bad |= pg < 0;
        }
        __syncwarp();
      } else {
        const uint32_t base = (uint32_t)(((long long)it.s * a.hkv + g) * a.cache.capacity + k0);
        for (int kk = lane; kk < it.nk; kk += 32) rows[kk] = base + kk;
      }
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        s_bad[sl] = bad ? 1 : 0;
        if (bad && a.status) atomicOr(a.status, CP_DEV_BOUNDS);
        s_items[sl * 2] = id;
        s_items[sl * 2 + 1] = it.nk;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[sl]);
    }
  }

  if (warp == kDecConsumers) {
    // ------------------------------------------------ issuer warp
    const unsigned char* kbase = static_cast<const unsigned char*>(a.k);
    const unsigned char* vbase = static_cast<const unsigned char*>(a.v);
    int t = 0;  // stages issued
    for (int j = 0;; ++j) {
      const int sl = j % NSL;
      if (!warp_wait(&ready[sl], (j / NSL) & 1, s_abort, a.status)) break;
      const int id = s_items[sl * 2];
      if (id < 0) {  // sentinel stage: ends the consumers
        const int st = t % NST, use = t / NST;
        if (use > 0 && !warp_wait(&empty[st], (use - 1) & 1, s_abort, a.status)) break;
        if (lane == 0) mbar_arrive(&full[st]);
        ++t;
        break;
      }
      DecItem it;
      dec_ids(a, id, nhb, it);
      it.nk = s_items[sl * 2 + 1];
      const uint32_t* rows = reinterpret_cast<const uint32_t*>(smem + L::rows) + sl * kDecodeSplit;
      const int ntl = (it.nk + SR - 1) / SR;
      bool alive = true;
      for (int tt = 0; tt < 2 * ntl; ++tt, ++t) {
        const int st = t % NST, use = t / NST;
        if (use > 0 && !warp_wait(&empty[st], (use - 1) & 1, s_abort, a.status)) {
          alive = false;
          break;
        }
        const int tl = tt < ntl ? tt : tt - ntl;
        const unsigned char* base = tt < ntl ? kbase : vbase;
        unsigned char* stage = smem + L::ring + st * kDecStageBytes;
#pragma unroll
        for (int rd = 0; rd < SR / 32; ++rd) {
          const int r = rd * 32 + lane;
          const int kk = tl * SR + r;
          const uint32_t row = kk < it.nk ? rows[kk] : kNoRow;
          const bool valid = row != kNoRow;
          const uint32_t prev = __shfl_up_sync(0xffffffffu, row, 1);
          const bool start = valid && (lane == 0 || prev == kNoRow || row != prev + 1);
          const uint32_t brk = __ballot_sync(0xffffffffu, start || !valid);
          const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
          if (lane == 0 && nvalid) mbar_expect_tx(&full[st], nvalid * L::kRow);
          __syncwarp();
          if (start) {
            const uint32_t later = lane == 31 ? 0u : (brk >> (lane + 1));
            const int len = later ? __ffs(later) : 32 - lane;
            bulk_load(stage + r * L::kRow, base + (long long)row * L::kRow, len * L::kRow, &full[st]);
          }
        }
        if (tt == 0 && lane == 0) {  // the item's q heads ride on its first stage
          const T* q = static_cast<const T*>(a.q) + ((long long)seq_row0(a.rows, it.s) * a.hq + it.hb * H) * D;
          mbar_expect_tx(&full[st], H * D * 2);
          bulk_load(smem + L::q + sl * H * D * 2, q, H * D * 2, &full[st]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      }
      if (!alive) break;
    }
    // Let every issued copy land before the CTA can exit.
    if (lane == 0) {
      for (int u = t - NST < 0 ? 0 : t - NST; u < t; ++u)
        if (!mbar_wait_drain(&full[u % NST], (u / NST) & 1) && a.status) atomicOr(a.status, CP_DEV_TIMEOUT);
    }
    return;
  }
  if (warp > kDecConsumers) return;

  // -------------------------------------------------- consumer warps
  const int sub = lane % LPK;
  const int r = warp * KPW + lane / LPK;  // this lane's row within a stage (K phase)
  // The LPK lanes of a row reduce their H partial dot products by halving:
  // at each xor level a lane keeps half of the heads it holds and adds its
  // partner's half, so after log2(LPK) levels lane `sub` holds the full dot
  // product of head hb (lanes sub and sub ^ 1 ... hold the same head).
  int hb = 0;
#pragma unroll
  for (int lvl = 0; (LPK >> (lvl + 1)) >= 1; ++lvl)
    if ((H >> lvl) > 1 && (lane & (LPK >> (lvl + 1)))) hb += (H >> lvl) / 2;
  constexpr int kHeadLanes = LPK / H;     // lanes of a row holding the same head
  const int subv = lane % LPV;
  const int rv = warp * RPW + lane / LPV;  // this lane's row within a V pass
  float (*sc)[kDecodeSplit] = reinterpret_cast<float (*)[kDecodeSplit]>(smem + L::sc);
  float (*red)[H][D] = reinterpret_cast<float (*)[H][D]>(smem + L::red);
  bool ok = true;
  int t = 0;
  for (int j = 0;; ++j) {
    const int sl = j % NSL;
    ok = ok && warp_wait(&full[t % NST], (t / NST) & 1, s_abort, a.status);
    const int id = ok ? s_items[sl * 2] : -1;
    if (consumers_sync_or(!ok || id < 0)) break;
    DecItem it;
    dec_ids(a, id, nhb, it);
    it.nk = s_items[sl * 2 + 1];
    const int ntl = (it.nk + SR - 1) / SR;
    const uint32_t* rows = reinterpret_cast<const uint32_t*>(smem + L::rows) + sl * kDecodeSplit;
    const bool bad = s_bad[sl] != 0;

    // q slices (chunks sub, sub + LPK) of the H heads, scaled into the log2 domain.
    float2 qv[H][8];
    {
      const unsigned char* qs = smem + L::q + sl * H * D * 2;
#pragma unroll
      for (int h = 0; h < H; ++h) {
        uint32_t w[8];
        lds_row(qs + h * D * 2, sub, LPK, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 f = unpack2<T>(w[e]);
          qv[h][e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
        }
      }
    }

    // ---- scores over the K stages
    float mx = -INFINITY;  // running max of this lane's head over its rows
    for (int tl = 0; tl < ntl; ++tl, ++t) {
      const int st = t % NST;
      if (tl > 0) ok = ok && warp_wait(&full[st], (t / NST) & 1, s_abort, a.status);
      if (!ok) continue;
#pragma unroll
      for (int kp = 0; kp < KPASS; ++kp) {
      const int kk = tl * SR + kp * KPP + r;
      uint32_t w[8];
      lds_row(smem + L::ring + st * kDecStageBytes + (kp * KPP + r) * L::kRow, sub, LPK, w);
      float2 acc[H];
#pragma unroll
      for (int h = 0; h < H; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 kf = unpack2<T>(w[e]);
#pragma unroll
        for (int h = 0; h < H; ++h) ffma2v(acc[h], qv[h][e], kf);
      }
      float v[H];
#pragma unroll
      for (int h = 0; h < H; ++h) v[h] = acc[h].x + acc[h].y;
#pragma unroll
      for (int lvl = 0; (LPK >> (lvl + 1)) >= 1; ++lvl) {
        const int o = LPK >> (lvl + 1);
        constexpr int kMaxH = H;
        const int nh = kMaxH >> lvl;
        if (nh > 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < nh / 2; ++i) {
            const float send = up ? v[i] : v[i + nh / 2];
            const float keep = up ? v[i + nh / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        } else {
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
      }
      if (kk < it.nk) {
        const float sv = (bad && rows[kk] == kNoRow) ? -INFINITY : v[0];
        if (sub % kHeadLanes == 0) sc[hb][kk] = sv;
        mx = fmaxf(mx, sv);
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // The warp's max per head: lanes holding the same head across the row groups.
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane < LPK && sub % kHeadLanes == 0) s_wmax[warp][hb] = mx;
    consumers_sync();

    // ---- split max / sum per query head (log2 domain): kDecConsumers / H
    // warps per head, each over an interleaved share of the split's keys.
    constexpr int WPH = kDecConsumers / H;
    if (ok) {
      const int h = warp % H, part = warp / H;
      float m = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) m = fmaxf(m, s_wmax[w][h]);
      float l = 0.f;
      for (int kk = part * 32 + lane; kk < it.nk; kk += 32 * WPH) {
        const float pr = (m == -INFINITY) ? 0.f : ex2_approx(sc[h][kk] - m);
        sc[h][kk] = pr;
        l += pr;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) s_psum[part][h] = l;
    }
    consumers_sync();

    // ---- p . V over the V stages: a group of LPV = D/8 lanes per row, one
    // 16-byte chunk per lane, so a quarter-warp again reads 128 contiguous bytes.
    float2 acc[H][4];
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
    for (int tl = 0; tl < ntl; ++tl, ++t) {
      const int st = t % NST;
      ok = ok && warp_wait(&full[st], (t / NST) & 1, s_abort, a.status);
      if (!ok) continue;
      const unsigned char* stage = smem + L::ring + st * kDecStageBytes;
#pragma unroll
      for (int p = 0; p < VPASS; ++p) {
        const int row = p * kDecConsumers * RPW + rv;
        const int kk = tl * SR + row;
        if (kk < it.nk && !(bad && rows[kk] == kNoRow)) {
          const uint4 c = *reinterpret_cast<const uint4*>(stage + row * L::kRow + subv * 16);
          const uint32_t w[4] = {c.x, c.y, c.z, c.w};
          float2 pp[H];
#pragma unroll
          for (int h = 0; h < H; ++h) pp[h] = make_float2(sc[h][kk], sc[h][kk]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 vf = unpack2<T>(w[e]);
#pragma unroll
            for (int h = 0; h < H; ++h) ffma2v(acc[h][e], pp[h], vf);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // Sum the RPW row slots of the warp (lanes with the same `subv`).
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int o = LPV; o < 32; o <<= 1) {
          acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, o);
          acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, o);
        }
    if (lane < LPV) {
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) *reinterpret_cast<float2*>(&red[warp][h][subv * 8 + 2 * e]) = acc[h][e];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&freed[sl]);  // done with this item's slot: q and row indices
    consumers_sync();
    if (!ok) continue;
    const int h0 = it.hb * H;
    const long long part_base = ((long long)it.s * a.hq + h0) * a.max_splits;
    for (int i = threadIdx.x; i < H * D; i += kDecConsumers * 32) {
      const int h = i / D, dd = i % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) v += red[w][h][dd];
      a.part_o[((part_base + (long long)h * a.max_splits) + it.split) * D + dd] = v;
    }
    if (threadIdx.x < H) {
      const int h = threadIdx.x;
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) m = fmaxf(m, s_wmax[w][h]);
#pragma unroll
      for (int p = 0; p < WPH; ++p) l += s_psum[p][h];
      const long long idx = (part_base + (long long)h * a.max_splits) + it.split;
      a.part_ml[idx * 2 + 0] = m;
      a.part_ml[idx * 2 + 1] = l;
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const AttnArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int s = blockIdx.x, h = blockIdx.y, dd = threadIdx.x;
  if (seq_rows(a.rows, s) != 1) return;
  const int past = a.past[s];
  const int n = past + 1;
  if (past < 0 || n > a.max_ctx) return;
  const int nsplit = (n + kDecodeSplit - 1) / kDecodeSplit;
  const long long base = ((long long)s * a.hq + h) * a.max_splits;
  float mx = -INFINITY;
  for (int i = 0; i < nsplit; ++i) mx = fmaxf(mx, a.part_ml[(base + i) * 2]);
  float acc = 0.f, l = 0.f;
  for (int i = 0; i < nsplit; ++i) {
    const float mi = a.part_ml[(base + i) * 2];
    const float w = (mi == -INFINITY) ? 0.f : ex2_approx(mi - mx);
    acc = fmaf(w, a.part_o[(base + i) * D + dd], acc);
    l = fmaf(w, a.part_ml[(base + i) * 2 + 1], l);
  }
  const float o = l > 0.f ? acc * (1.f / l) : 0.f;
  T* out = static_cast<T*>(a.out);
  out[((long long)seq_row0(a.rows, s) * a.hq + h) * D + dd] = from_float<T>(o);
}

template <typename T, int D, int H>
cudaError_t launch_decode_t(const AttnArgs& a, int* counter, cudaStream_t st) {
  constexpr int smem = DecSmem<D, H>::bytes;
  // The dynamic shared-memory limit is a per-device function attribute: raise
  // it once per device, so later calls (including ones being captured into a
  // CUDA graph) only launch.
  static std::atomic<uint64_t> ready_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(decode_split_kernel<T, D, H>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ready_mask.fetch_or(bit, std::memory_order_release);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)a.max_splits * a.rows.num_seqs * (a.hq / H);
  if (items >= (1ll << 31) - (1ll << 20)) return cudaErrorInvalidValue;
  // Row indices are 32-bit: the cache must hold fewer than 2^32 - 1 rows.
  const long long cache_rows = a.cache.kind == CP_CACHE_PAGED
                                   ? (long long)a.cache.num_pages * a.hkv * a.cache.page_size
                                   : (long long)a.rows.num_seqs * a.hkv * a.cache.capacity;
  if (cache_rows >= (long long)kNoRow) return cudaErrorInvalidValue;
  const int grid = (int)(items < (long long)sms * kDecCtasPerSm ? items : (long long)sms * kDecCtasPerSm);
  e = cudaMemsetAsync(counter, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_split_kernel<T, D, H>, dim3(grid), dim3((kDecConsumers + 2) * 32), smem, st, a, counter);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_combine_kernel<T, D>, dim3(a.rows.num_seqs, a.hq), dim3(D), 0, st, a);
}

// Query heads per CTA: the whole GQA group up to 4 (a group of 8 takes two
// CTAs, which read the same K/V rows, the second mostly from L2).
template <typename T, int D>
cudaError_t launch_decode_d(const AttnArgs& a, int* counter, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_decode_t<T, D, 1>(a, counter, st);
    case 2: return launch_decode_t<T, D, 2>(a, counter, st);
    case 4:
    case 8: return launch_decode_t<T, D, 4>(a, counter, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_supported(int d, int group, int dtype) {
  return (d == 64 || d == 128) && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == CP_BF16 || dtype == CP_F16);
}

cudaError_t launch_decode(const AttnArgs& a, int dtype, int* counter, cudaStream_t st) {
  if (a.rows.num_seqs == 0 || a.max_splits == 0) return cudaSuccess;
  if (dtype == CP_BF16) return a.d == 64 ? launch_decode_d<__nv_bfloat16, 64>(a, counter, st)
                                         : launch_decode_d<__nv_bfloat16, 128>(a, counter, st);
  return a.d == 64 ? launch_decode_d<__half, 64>(a, counter, st) : launch_decode_d<__half, 128>(a, counter, st);
}

}  // namespace cp
