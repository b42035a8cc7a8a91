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

constexpr int kDecConsumers = 4;            // consumer warps per CTA (plus one producer warp)
constexpr int kDecStageKeys = 32;           // K or V rows per ring stage
constexpr int kDecRingBytes = 48 * 1024;    // ring of stages: 6 stages at D = 128, 12 at D = 64

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
  static constexpr int kRow = D * 2;                       // bytes of one K or V row
  static constexpr int kStageBytes = kDecStageKeys * kRow;
  static constexpr int kStages = kDecRingBytes / kStageBytes;
  static constexpr int ring = 0;
  static constexpr int full = ring + kDecRingBytes;        // uint64 [kStages]
  static constexpr int empty = full + 8 * kStages;         // uint64 [kStages]
  static constexpr int off = empty + 8 * kStages;          // long long [kDecodeSplit]
  static constexpr int sc = off + 8 * kDecodeSplit;        // float [H][kDecodeSplit]
  static constexpr int ml = sc + 4 * H * kDecodeSplit;     // float [2][H]
  static constexpr int flags = ml + 8 * H;                 // int abort, bad
  static constexpr int bytes = flags + 16;
  static_assert(kDecConsumers * H * D * 4 <= kDecRingBytes, "reduction buffer aliases the ring");
};

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDecConsumers * 32) : "memory"); }

// Row j of a staged tile, as the two 16-byte chunks c0 = sub and c1 = sub + LPK.
__device__ __forceinline__ void lds_row(const unsigned char* row, int sub, int lpk, uint32_t (&w)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(row + sub * 16);
  const uint4 b = *reinterpret_cast<const uint4*>(row + (sub + lpk) * 16);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// One CTA per (split of kDecodeSplit keys, H query heads of one KV group,
// sequence).  Warp kDecConsumers is the producer: it resolves the split's key
// rows to cache offsets once, then streams the split's K rows and then its V
// rows through a ring of kDecStageKeys-row stages with bulk copies (one copy
// per run of contiguous rows: a whole stage for a contiguous cache, one page
// per copy for a paged one), so the bytes in flight are bounded by shared
// memory, not by registers.  Warps 0..kDecConsumers-1 consume: a group of
// LPK = D/16 lanes takes one row, 16 elements per lane (chunks sub and
// sub+LPK, so a quarter-warp reads 128 contiguous bytes), with packed fp32x2
// FMAs; scores go to shared memory, the split's max and sum are taken in the
// log2 domain, then the V stages are consumed and the unnormalised partial
// output written.
template <typename T, int D, int H>
__global__ void __launch_bounds__((kDecConsumers + 1) * 32) decode_split_kernel(const AttnArgs a) {
  using L = DecSmem<D, H>;
  constexpr int LPK = D / 16;                 // lanes per row
  constexpr int KPW = 32 / LPK;               // rows per warp per pass
  constexpr int KPP = kDecConsumers * KPW;    // rows per pass
  constexpr int PASSES = kDecStageKeys / KPP;
  constexpr int NST = L::kStages;
  static_assert(kDecStageKeys % KPP == 0 && kDecStageKeys == 32, "one producer lane per staged row");
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::empty);
  long long* s_off = reinterpret_cast<long long*>(smem + L::off);
  float (*sc)[kDecodeSplit] = reinterpret_cast<float (*)[kDecodeSplit]>(smem + L::sc);
  float* s_m = reinterpret_cast<float*>(smem + L::ml);
  float* s_l = s_m + H;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::flags);
  volatile int* s_bad = s_abort + 1;

  const int split = blockIdx.x, hb = blockIdx.y, s = blockIdx.z;
  if (seq_rows(a.rows, s) != 1) return;
  const int past = a.past[s];
  const int n = past + 1;
  if (past < 0 || n > a.max_ctx) {
    if (a.status && threadIdx.x == 0 && split == 0 && hb == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int k0 = split * kDecodeSplit;
  if (k0 >= n) return;
  const int nk = min(n - k0, kDecodeSplit);
  const int nt = (nk + kDecStageKeys - 1) / kDecStageKeys;  // stages per phase
  const int h0 = hb * H;                                    // first query head
  const int g = h0 / a.group;                               // its KV head

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecConsumers);
    }
    *s_abort = 0;
    *s_bad = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kDecConsumers) {
    // ------------------------------------------------ producer warp
    bool bad = false;
    for (int kk = lane; kk < nk; kk += 32) {
      const long long off = key_offset(a.cache, a.hkv, D, s, g, k0 + kk);
      s_off[kk] = off;
      bad |= off < 0;
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) {
        *s_bad = 1;
        if (a.status) atomicOr(a.status, CP_DEV_BOUNDS);
      }
    }
    __syncwarp();
    const unsigned char* base[2] = {static_cast<const unsigned char*>(a.k), static_cast<const unsigned char*>(a.v)};
    int issued = 0;
    for (int t = 0; t < 2 * nt; ++t) {
      const int st = t % NST, use = t / NST;
      if (use > 0 && !warp_wait(&empty[st], (use - 1) & 1, s_abort, a.status)) break;
      const int tl = t < nt ? t : t - nt;
      const int kk = tl * kDecStageKeys + lane;
      const long long off = kk < nk ? s_off[kk] : -1;
      const bool valid = off >= 0;
      const long long prev = __shfl_up_sync(0xffffffffu, off, 1);
      const bool start = valid && (lane == 0 || prev < 0 || off != prev + D);
      const uint32_t brk = __ballot_sync(0xffffffffu, start || !valid);
      const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
      if (lane == 0) mbar_expect_tx(&full[st], nvalid * L::kRow);
      __syncwarp();
      if (start) {
        const uint32_t later = lane == 31 ? 0u : (brk >> (lane + 1));
        const int len = later ? __ffs(later) : 32 - lane;
        bulk_load(smem + L::ring + st * L::kStageBytes + lane * L::kRow,
                  base[t < nt ? 0 : 1] + off * (long long)sizeof(T), len * L::kRow, &full[st]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      issued = t + 1;
    }
    // Let every issued copy land before the CTA can exit.
    if (lane == 0) {
      for (int t = issued - NST < 0 ? 0 : issued - NST; t < issued; ++t)
        if (!mbar_wait_drain(&full[t % NST], (t / NST) & 1) && a.status) atomicOr(a.status, CP_DEV_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------- consumer warps
  const int sub = lane % LPK;
  const int slot = warp * KPW + lane / LPK;
  bool ok = true;

  // q slices (chunks sub, sub + LPK) of the H heads, scaled into the log2 domain.
  float2 qv[H][8];
  {
    const T* q = static_cast<const T*>(a.q) + ((long long)seq_row0(a.rows, s) * a.hq + h0) * D;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      const uint4 r0 = *reinterpret_cast<const uint4*>(q + h * D + sub * 8);
      const uint4 r1 = *reinterpret_cast<const uint4*>(q + h * D + (sub + LPK) * 8);
      const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 f = unpack2<T>(w[e]);
        qv[h][e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
      }
    }
  }

  // ---- scores over the K stages
  for (int t = 0; t < nt; ++t) {
    const int st = t % NST;
    ok = ok && warp_wait(&full[st], (t / NST) & 1, s_abort, a.status);
    if (ok) {
      const bool bad = *s_bad != 0;
      const unsigned char* stage = smem + L::ring + st * L::kStageBytes;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int r = p * KPP + slot;
        const int kk = t * kDecStageKeys + r;
        uint32_t w[8];
        lds_row(stage + r * L::kRow, sub, LPK, w);
        float2 acc[H];
#pragma unroll
        for (int h = 0; h < H; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 kf = unpack2<T>(w[e]);
#pragma unroll
          for (int h = 0; h < H; ++h) ffma2v(acc[h], qv[h][e], kf);
        }
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float v = acc[h].x + acc[h].y;
#pragma unroll
          for (int o = LPK / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (sub == 0 && kk < nk) sc[h][kk] = (bad && s_off[kk] < 0) ? -INFINITY : v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  consumers_sync();

  // ---- split max / sum per query head (log2 domain)
  if (ok) {
    for (int h = warp; h < H; h += kDecConsumers) {
      float m = -INFINITY;
      for (int kk = lane; kk < nk; kk += 32) m = fmaxf(m, sc[h][kk]);
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float l = 0.f;
      for (int kk = lane; kk < nk; kk += 32) {
        const float pr = (m == -INFINITY) ? 0.f : ex2_approx(sc[h][kk] - m);
        sc[h][kk] = pr;
        l += pr;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) {
        s_m[h] = m;
        s_l[h] = l;
      }
    }
  }
  consumers_sync();

  // ---- p . V over the V stages
  float2 acc[H][8];
#pragma unroll
  for (int h = 0; h < H; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = make_float2(0.f, 0.f);
  for (int t = 0; t < nt; ++t) {
    const int st = (nt + t) % NST;
    ok = ok && warp_wait(&full[st], ((nt + t) / NST) & 1, s_abort, a.status);
    if (ok) {
      const bool bad = *s_bad != 0;
      const unsigned char* stage = smem + L::ring + st * L::kStageBytes;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int r = p * KPP + slot;
        const int kk = t * kDecStageKeys + r;
        if (kk < nk && !(bad && s_off[kk] < 0)) {
          uint32_t w[8];
          lds_row(stage + r * L::kRow, sub, LPK, w);
          float2 pp[H];
#pragma unroll
          for (int h = 0; h < H; ++h) pp[h] = make_float2(sc[h][kk], sc[h][kk]);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 vf = unpack2<T>(w[e]);
#pragma unroll
            for (int h = 0; h < H; ++h) ffma2v(acc[h][e], pp[h], vf);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  // Sum the KPW row slots of the warp (lanes with the same `sub`).
#pragma unroll
  for (int h = 0; h < H; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1) {
        acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, o);
        acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, o);
      }
  consumers_sync();  // every warp is done with the ring, which now holds the reduction
  float (*red)[H][D] = reinterpret_cast<float (*)[H][D]>(smem + L::ring);
  if (lane < LPK) {
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        red[warp][h][sub * 8 + 2 * e] = acc[h][e].x;
        red[warp][h][sub * 8 + 2 * e + 1] = acc[h][e].y;
        red[warp][h][(sub + LPK) * 8 + 2 * e] = acc[h][e + 4].x;
        red[warp][h][(sub + LPK) * 8 + 2 * e + 1] = acc[h][e + 4].y;
      }
  }
  consumers_sync();
  if (!ok || *s_abort) return;
  const long long part_base = ((long long)s * a.hq + h0) * a.max_splits;
  for (int i = threadIdx.x; i < H * D; i += kDecConsumers * 32) {
    const int h = i / D, dd = i % D;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDecConsumers; ++w) v += red[w][h][dd];
    a.part_o[((part_base + (long long)h * a.max_splits) + split) * D + dd] = v;
  }
  if (threadIdx.x < H) {
    const long long idx = (part_base + (long long)threadIdx.x * a.max_splits) + split;
    a.part_ml[idx * 2 + 0] = s_m[threadIdx.x];
    a.part_ml[idx * 2 + 1] = s_l[threadIdx.x];
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const AttnArgs a) {
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
cudaError_t launch_decode_t(const AttnArgs& a, cudaStream_t st) {
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
  dim3 grid(a.max_splits, a.hq / H, a.rows.num_seqs);
  decode_split_kernel<T, D, H><<<grid, (kDecConsumers + 1) * 32, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<T, D><<<dim3(a.rows.num_seqs, a.hq), D, 0, st>>>(a);
  return cudaGetLastError();
}

// Query heads per CTA: the whole GQA group up to 4 (a group of 8 takes two
// CTAs, which read the same K/V rows, the second mostly from L2).
template <typename T, int D>
cudaError_t launch_decode_d(const AttnArgs& a, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_decode_t<T, D, 1>(a, st);
    case 2: return launch_decode_t<T, D, 2>(a, st);
    case 4:
    case 8: return launch_decode_t<T, D, 4>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_supported(int d, int group, int dtype) {
  return (d == 64 || d == 128) && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == CP_BF16 || dtype == CP_F16);
}

cudaError_t launch_decode(const AttnArgs& a, int dtype, cudaStream_t st) {
  if (a.rows.num_seqs == 0 || a.max_splits == 0) return cudaSuccess;
  if (dtype == CP_BF16) return a.d == 64 ? launch_decode_d<__nv_bfloat16, 64>(a, st)
                                         : launch_decode_d<__nv_bfloat16, 128>(a, st);
  return a.d == 64 ? launch_decode_d<__half, 64>(a, st) : launch_decode_d<__half, 128>(a, st);
}

}  // namespace cp
