// decode.cu -- single-row (decode) attention on the memory-bound split-KV path.
//
// A decode row reads its sequence's whole K/V once and does ~1 FLOP per byte
// (Ultralytics glossary "Chunked Prefill", "Prefill, decode and generation
// stalls": decode is memory-bandwidth bound), so this path is built to keep
// HBM streaming: K and V rows go straight from global memory into registers
// with coalesced 16-byte loads, and the few FLOPs per byte run on the warp-
// level tensor-core MMA (m16n8k16, fp32 accumulate), which spends one
// instruction where fp32 FMAs and lane reductions would spend dozens.
//
// decode_split_kernel: one CTA per (split of 512 keys, KV head, sequence), four
//   warps of 128 keys each.  The query rows of the sequence's k rows (k = 1 for
//   decode; a short chunk -- k draft tokens verified in one pass -- when
//   k * G <= 16) times the GQA group's G query heads ride in the MMA's N
//   dimension: NF fragments of 8 columns, column c <-> (row c / G, head c % G),
//   columns past k * G zero.  Every row reads the same K/V registers; row r
//   masks the keys after its own position past + r.
//   Scores: S^T[16 keys x 8 heads] = K[16 keys x D] Q^T, as D/16 MMAs per
//   16-key tile.  Lane (g, q) (g = lane / 4, q = lane % 4) loads keys g and
//   g + 8 of the tile, 16-byte chunks q, q + 4, ...; under the head-dimension
//   order that maps MMA column pair (2q, 2q + 1) of slice (j, u) to elements
//   4u, 4u + 1 of chunk q + 4j (and columns 2q + 8, 2q + 9 to 4u + 2, 4u + 3),
//   those loaded registers ARE the A fragments, and the query is loaded into
//   B fragments in the same order.  The dot product does not depend on the
//   order in which the head dimension is summed.
//   Softmax: each warp takes its own max per head over its 128 keys (log2
//   domain), writes P (16-bit) to shared memory and sums it.
//   Output: O^T[16 dims x 8 heads] += V^T[16 dims x 16 keys] P^T.  Lane (g, q)
//   loads keys 2q, 2q + 1, 2q + 8, 2q + 9 of the tile, chunks g, g + 8, ...;
//   byte permutes pair up the same element of two keys, which is the A
//   fragment of the 16-row block of dims {8c + 2i, 8c + 2i + 1 : c = g + 8m}.
//   The four warps' partials are merged in warp order with their maxima, and
//   the split's unnormalised output and (max, sum) are written for the
//   combine kernel.
// decode_combine_kernel: merges a row's split partials in split order
//   (log-sum-exp), so the result depends only on the row's own context.
#include <cmath>
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kDecWarps = 4;                          // warps per CTA
constexpr int kDecWarpKeys = kDecodeSplit / kDecWarps;  // 128 keys per warp
constexpr int kDecTiles = kDecWarpKeys / 16;          // 16-key MMA tiles per warp
constexpr int kDecCols = 8;                           // MMA N per fragment: (row, head) columns, zero-padded
constexpr int kPStride = kDecWarpKeys + 8;            // 16-bit P row stride: conflict-free fragment reads
static_assert(kDecWarps * kDecWarpKeys == kDecodeSplit, "the warps cover a split");

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

template <typename T>
__device__ __forceinline__ uint16_t bits16(float x) {
  const T h = from_float<T>(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// 16 bytes from global memory that is read once: no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// D (16x8, fp32) += A (16x16, row) * B (16x8, col), 16-bit inputs.
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecWarps * 32, 4) decode_split_kernel(const AttnArgs a) {
  constexpr int NJ = D / 32;  // score phase: chunks per lane per key
  constexpr int NM = D / 64;  // output phase: chunks per lane per key
  constexpr int kRowBytes = D * 2;
  __shared__ __align__(16) uint16_t sP[kDecWarps][kDecCols][kPStride];
  __shared__ __align__(16) float sO[kDecWarps][kDecCols][D];
  __shared__ float sM[kDecWarps][kDecCols], sL[kDecWarps][kDecCols];

  pdl_launch_dependents();
  const int split = blockIdx.x % a.max_splits, s = blockIdx.x / a.max_splits, gk = blockIdx.y;
  pdl_wait();  // everything below reads what earlier kernels wrote
  // One-call chunk: `past` is a copy of the lengths, so one CTA may advance them at once.
  if (a.commit_lens && !a.ticket && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < a.rows.num_seqs; i += blockDim.x) a.commit_lens[i] += a.commit_add;
  if (seq_rows(a.rows, s) != 1) return;
  const int past = a.past[s];
  const int n = past + 1;
  if (past < 0 || n > a.max_ctx) {
    if (a.status && split == 0 && gk == 0 && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int k0 = split * kDecodeSplit;
  if (k0 >= n) return;
  const int nk = min(n - k0, kDecodeSplit);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, q4 = lane & 3;
  const int G = a.group;
  const int kw = warp * kDecWarpKeys;                   // the warp's first key in the split
  const int nkw = max(0, min(nk - kw, kDecWarpKeys));   // its valid keys
  const int ntile = (nkw + 15) / 16;
  const bool paged = a.cache.kind == CP_CACHE_PAGED;
  const int ps = a.cache.page_size;

  // Page of each of the warp's tiles (a page holds whole 16-key tiles).
  int pgv = -1;
  if (paged && lane < ntile) {
    const int blk = (k0 + kw + 16 * lane) / ps;
    int pg = blk < a.cache.max_blocks ? a.cache.block_table[(long long)s * a.cache.max_blocks + blk] : -1;
    if (pg < 0 || pg >= a.cache.num_pages) {
      if (a.status) atomicOr(a.status, CP_DEV_BOUNDS);
      pg = -1;
    }
    pgv = pg;
  }
  // Byte offset of row 0 of tile t in the K (or V) cache, or -1 (tile's page invalid).
  auto tile_off = [&](int t) -> long long {
    if (paged) {
      const int pg = __shfl_sync(0xffffffffu, pgv, t);
      if (pg < 0) return -1;
      return (((long long)pg * a.hkv + gk) * ps + (k0 + kw + 16 * t) % ps) * kRowBytes;
    }
    return (((long long)s * a.hkv + gk) * a.cache.capacity + k0 + kw + 16 * t) * kRowBytes;
  };
  const unsigned char* kbase = static_cast<const unsigned char*>(a.k);
  const unsigned char* vbase = static_cast<const unsigned char*>(a.v);

  // Query B fragments: head g8 (zero past the group), chunks q4 + 4j.
  uint4 qf[NJ];
  {
    const bool hv = g8 < G;
    const unsigned char* qrow =
        static_cast<const unsigned char*>(a.q) + (((long long)seq_row0(a.rows, s) * a.hq + gk * G + g8) * D) * 2;
#pragma unroll
    for (int j = 0; j < NJ; ++j) qf[j] = hv ? *reinterpret_cast<const uint4*>(qrow + (q4 + 4 * j) * 16) : make_uint4(0, 0, 0, 0);
  }

  // ---- scores: keys g8 and g8 + 8 of each tile, heads 2q4 and 2q4 + 1
  float sc[kDecTiles][4];
  auto load_k = [&](int t, uint4 (&kr)[2][NJ]) {
    const long long off = t < ntile ? tile_off(t) : -1;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int key = 16 * t + g8 + 8 * r;
      const bool ok = off >= 0 && key < nkw;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        kr[r][j] = ok ? ldg_stream(kbase + off + (g8 + 8 * r) * kRowBytes + (q4 + 4 * j) * 16) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 kb[2][2][NJ];
  load_k(0, kb[0]);
  float mx0 = -INFINITY, mx1 = -INFINITY;
  const bool h0v = 2 * q4 < G, h1v = 2 * q4 + 1 < G;
#pragma unroll
  for (int t = 0; t < kDecTiles; ++t) {
    if (t + 1 < kDecTiles) load_k(t + 1, kb[(t + 1) & 1]);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4 (&kr)[2][NJ] = kb[t & 1];
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
      for (int u = 0; u < 2; ++u)
        mma16816<T>(c, word(kr[0][j], 2 * u), word(kr[1][j], 2 * u), word(kr[0][j], 2 * u + 1),
                    word(kr[1][j], 2 * u + 1), word(qf[j], 2 * u), word(qf[j], 2 * u + 1));
    const long long off = t < ntile ? tile_off(t) : -1;
    const bool k0v = off >= 0 && 16 * t + g8 < nkw, k1v = off >= 0 && 16 * t + g8 + 8 < nkw;
    sc[t][0] = (k0v && h0v) ? c[0] * a.scale_log2 : -INFINITY;
    sc[t][1] = (k0v && h1v) ? c[1] * a.scale_log2 : -INFINITY;
    sc[t][2] = (k1v && h0v) ? c[2] * a.scale_log2 : -INFINITY;
    sc[t][3] = (k1v && h1v) ? c[3] * a.scale_log2 : -INFINITY;
    mx0 = fmaxf(mx0, fmaxf(sc[t][0], sc[t][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[t][1], sc[t][3]));
  }
  // The first V tile is in flight while the softmax runs.
  auto load_v = [&](int t, uint4 (&vr)[4][NM]) {
    const long long off = t < ntile ? tile_off(t) : -1;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int kt = 2 * q4 + (r & 1) + 8 * (r >> 1);  // key within the tile: 2q, 2q+1, 2q+8, 2q+9
      const bool ok = off >= 0 && 16 * t + kt < nkw;
#pragma unroll
      for (int m = 0; m < NM; ++m)
        vr[r][m] = ok ? ldg_stream(vbase + off + kt * kRowBytes + (g8 + 8 * m) * 16) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 vb[2][4][NM];
  if (ntile > 0) load_v(0, vb[0]);
  // The warp's max per head: over the eight lanes g8 that share q4.
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  // P (16-bit) for the output MMAs, and its sum in fp32.
  float l0 = 0.f, l1 = 0.f;
  uint16_t(*pw)[kPStride] = sP[warp];
#pragma unroll
  for (int t = 0; t < kDecTiles; ++t) {
    const float p0 = mx0 == -INFINITY ? 0.f : ex2_approx(sc[t][0] - mx0);
    const float p1 = mx1 == -INFINITY ? 0.f : ex2_approx(sc[t][1] - mx1);
    const float p2 = mx0 == -INFINITY ? 0.f : ex2_approx(sc[t][2] - mx0);
    const float p3 = mx1 == -INFINITY ? 0.f : ex2_approx(sc[t][3] - mx1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    pw[2 * q4][16 * t + g8] = bits16<T>(p0);
    pw[2 * q4 + 1][16 * t + g8] = bits16<T>(p1);
    pw[2 * q4][16 * t + g8 + 8] = bits16<T>(p2);
    pw[2 * q4 + 1][16 * t + g8 + 8] = bits16<T>(p3);
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  __syncwarp();

  // ---- output: dims 8(g8 + 8m) + 2i2 (+1) for heads 2q4, 2q4 + 1
  float o[NM * 4][4];
#pragma unroll
  for (int b = 0; b < NM * 4; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.f;
#pragma unroll
  for (int t = 0; t < kDecTiles; ++t) {
    if (t < ntile) {
      if (t + 1 < ntile) load_v(t + 1, vb[(t + 1) & 1]);
      const uint4 (&vr)[4][NM] = vb[t & 1];
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&pw[g8][16 * t + 2 * q4]);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&pw[g8][16 * t + 2 * q4 + 8]);
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const uint32_t x0 = word(vr[0][m], i2), x1 = word(vr[1][m], i2);
          const uint32_t x2 = word(vr[2][m], i2), x3 = word(vr[3][m], i2);
          mma16816<T>(o[m * 4 + i2], __byte_perm(x0, x1, 0x5410), __byte_perm(x0, x1, 0x7632),
                      __byte_perm(x2, x3, 0x5410), __byte_perm(x2, x3, 0x7632), b0, b1);
        }
    }
  }
  // The warp's partial: heads 2q4, 2q4 + 1 (those of the group), rows of dims.
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      const int d0 = 8 * (g8 + 8 * m) + 2 * i2;
      if (h0v) *reinterpret_cast<float2*>(&sO[warp][2 * q4][d0]) = make_float2(o[m * 4 + i2][0], o[m * 4 + i2][2]);
      if (h1v) *reinterpret_cast<float2*>(&sO[warp][2 * q4 + 1][d0]) = make_float2(o[m * 4 + i2][1], o[m * 4 + i2][3]);
    }
  if (g8 == 0) {
    sM[warp][2 * q4] = mx0;
    sL[warp][2 * q4] = l0;
    sM[warp][2 * q4 + 1] = mx1;
    sL[warp][2 * q4 + 1] = l1;
  }
  __syncthreads();

  // ---- the split's partial: the warps' partials merged in warp order
  const long long part_base = ((long long)s * a.hq + gk * G) * a.max_splits;
  for (int i = threadIdx.x; i < G * D; i += kDecWarps * 32) {
    const int h = i / D, dd = i % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, sM[w][h]);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (sM[w][h] != -INFINITY) v += ex2_approx(sM[w][h] - m) * sO[w][h][dd];
    a.part_o[((part_base + (long long)h * a.max_splits) + split) * D + dd] = v;
  }
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, sM[w][h]);
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (sM[w][h] != -INFINITY) l += ex2_approx(sM[w][h] - m) * sL[w][h];
    const long long idx = (part_base + (long long)h * a.max_splits) + split;
    a.part_ml[idx * 2 + 0] = m;
    a.part_ml[idx * 2 + 1] = l;
  }
}

// The same for k > 1 rows per sequence (a short chunk, k * G <= 16): NF
// fragments of 8 (row, head) columns; row r masks the keys after past + r.
template <typename T, int D, int NF>
__global__ void __launch_bounds__(kDecWarps * 32, NF == 1 ? 4 : 3) decode_rows_kernel(const AttnArgs a) {
  constexpr int NJ = D / 32;  // score phase: chunks per lane per key
  constexpr int NM = D / 64;  // output phase: chunks per lane per key
  constexpr int NC = kDecCols * NF;  // (row, head) columns
  constexpr int kRowBytes = D * 2;
  __shared__ __align__(16) uint16_t sP[kDecWarps][NC][kPStride];
  __shared__ __align__(16) float sO[kDecWarps][NC][D];
  __shared__ float sM[kDecWarps][NC], sL[kDecWarps][NC];

  pdl_launch_dependents();
  const int split = blockIdx.x % a.max_splits, s = blockIdx.x / a.max_splits, gk = blockIdx.y;
  pdl_wait();  // everything below reads what earlier kernels wrote
  // One-call chunk: `past` is a copy of the lengths, so one CTA may advance them at once.
  if (a.commit_lens && !a.ticket && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < a.rows.num_seqs; i += blockDim.x) a.commit_lens[i] += a.commit_add;
  const int kr = a.dec_rows;  // rows per sequence on this path
  if (seq_rows(a.rows, s) != kr) return;
  const int past = a.past[s];
  const int n = past + kr;  // keys, including this call's rows
  if (past < 0 || n > a.max_ctx) {
    if (a.status && split == 0 && gk == 0 && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int k0 = split * kDecodeSplit;
  if (k0 >= n) return;
  const int nk = min(n - k0, kDecodeSplit);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, q4 = lane & 3;
  const int G = a.group;
  const int kw = warp * kDecWarpKeys;                   // the warp's first key in the split
  const int nkw = max(0, min(nk - kw, kDecWarpKeys));   // its valid keys
  const int ntile = (nkw + 15) / 16;
  const bool paged = a.cache.kind == CP_CACHE_PAGED;
  const int ps = a.cache.page_size;

  // Page of each of the warp's tiles (a page holds whole 16-key tiles).
  int pgv = -1;
  if (paged && lane < ntile) {
    const int blk = (k0 + kw + 16 * lane) / ps;
    int pg = blk < a.cache.max_blocks ? a.cache.block_table[(long long)s * a.cache.max_blocks + blk] : -1;
    if (pg < 0 || pg >= a.cache.num_pages) {
      if (a.status) atomicOr(a.status, CP_DEV_BOUNDS);
      pg = -1;
    }
    pgv = pg;
  }
  // Byte offset of row 0 of tile t in the K (or V) cache, or -1 (tile's page invalid).
  auto tile_off = [&](int t) -> long long {
    if (paged) {
      const int pg = __shfl_sync(0xffffffffu, pgv, t);
      if (pg < 0) return -1;
      return (((long long)pg * a.hkv + gk) * ps + (k0 + kw + 16 * t) % ps) * kRowBytes;
    }
    return (((long long)s * a.hkv + gk) * a.cache.capacity + k0 + kw + 16 * t) * kRowBytes;
  };
  const unsigned char* kbase = static_cast<const unsigned char*>(a.k);
  const unsigned char* vbase = static_cast<const unsigned char*>(a.v);

  // Query B fragments: column 8f + g8 = (row r, head h) (zero past k * G), chunks q4 + 4j.
  const int ncols = kr * G;
  uint4 qf[NF][NJ];
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const int c = kDecCols * f + g8;
    const bool cv = c < ncols;
    const int r = cv ? c / G : 0, h = cv ? c % G : 0;
    const unsigned char* qrow = static_cast<const unsigned char*>(a.q) +
                                (((long long)(seq_row0(a.rows, s) + r) * a.hq + gk * G + h) * D) * 2;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      qf[f][j] = cv ? *reinterpret_cast<const uint4*>(qrow + (q4 + 4 * j) * 16) : make_uint4(0, 0, 0, 0);
  }

  // ---- scores: keys g8 and g8 + 8 of each tile, columns 8f + 2q4 and 8f + 2q4 + 1
  float sc[kDecTiles][NF][4];
  auto load_k = [&](int t, uint4 (&kr)[2][NJ]) {
    const long long off = t < ntile ? tile_off(t) : -1;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int key = 16 * t + g8 + 8 * r;
      const bool ok = off >= 0 && key < nkw;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        kr[r][j] = ok ? ldg_stream(kbase + off + (g8 + 8 * r) * kRowBytes + (q4 + 4 * j) * 16) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 kb[2][2][NJ];
  load_k(0, kb[0]);
  float mx[NF][2];
  int lim[NF][2];  // last key index (within the split) that column 8f + 2q4 + e may see; -1: none
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[f][e] = -INFINITY;
      const int c = kDecCols * f + 2 * q4 + e;
      lim[f][e] = c < ncols ? past + c / G - k0 : -1;  // row r sees keys up to past + r
    }
#pragma unroll
  for (int t = 0; t < kDecTiles; ++t) {
    if (t + 1 < kDecTiles) load_k(t + 1, kb[(t + 1) & 1]);
    const uint4 (&kv)[2][NJ] = kb[t & 1];
    const long long off = t < ntile ? tile_off(t) : -1;
    const int kt0 = 16 * t + g8;  // keys kt0, kt0 + 8 of the warp
    const bool k0v = off >= 0 && kt0 < nkw, k1v = off >= 0 && kt0 + 8 < nkw;
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u)
          mma16816<T>(c, word(kv[0][j], 2 * u), word(kv[1][j], 2 * u), word(kv[0][j], 2 * u + 1),
                      word(kv[1][j], 2 * u + 1), word(qf[f][j], 2 * u), word(qf[f][j], 2 * u + 1));
      const bool v00 = kw + kt0 <= lim[f][0], v01 = kw + kt0 <= lim[f][1];
      const bool v10 = kw + kt0 + 8 <= lim[f][0], v11 = kw + kt0 + 8 <= lim[f][1];
      sc[t][f][0] = (k0v && v00) ? c[0] * a.scale_log2 : -INFINITY;
      sc[t][f][1] = (k0v && v01) ? c[1] * a.scale_log2 : -INFINITY;
      sc[t][f][2] = (k1v && v10) ? c[2] * a.scale_log2 : -INFINITY;
      sc[t][f][3] = (k1v && v11) ? c[3] * a.scale_log2 : -INFINITY;
      mx[f][0] = fmaxf(mx[f][0], fmaxf(sc[t][f][0], sc[t][f][2]));
      mx[f][1] = fmaxf(mx[f][1], fmaxf(sc[t][f][1], sc[t][f][3]));
    }
  }
  // The first V tile is in flight while the softmax runs.
  auto load_v = [&](int t, uint4 (&vr)[4][NM]) {
    const long long off = t < ntile ? tile_off(t) : -1;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int kt = 2 * q4 + (r & 1) + 8 * (r >> 1);  // key within the tile: 2q, 2q+1, 2q+8, 2q+9
      const bool ok = off >= 0 && 16 * t + kt < nkw;
#pragma unroll
      for (int m = 0; m < NM; ++m)
        vr[r][m] = ok ? ldg_stream(vbase + off + kt * kRowBytes + (g8 + 8 * m) * 16) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 vb[2][4][NM];
  if (ntile > 0) load_v(0, vb[0]);
  // The warp's max per column: over the eight lanes g8 that share q4.
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx[f][0] = fmaxf(mx[f][0], __shfl_xor_sync(0xffffffffu, mx[f][0], o));
      mx[f][1] = fmaxf(mx[f][1], __shfl_xor_sync(0xffffffffu, mx[f][1], o));
    }
  // P (16-bit) for the output MMAs, and its sum in fp32.
  float l[NF][2];
  uint16_t(*pw)[kPStride] = sP[warp];
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    l[f][0] = l[f][1] = 0.f;
    const int c0 = kDecCols * f + 2 * q4;
#pragma unroll
    for (int t = 0; t < kDecTiles; ++t) {
      const float p0 = mx[f][0] == -INFINITY ? 0.f : ex2_approx(sc[t][f][0] - mx[f][0]);
      const float p1 = mx[f][1] == -INFINITY ? 0.f : ex2_approx(sc[t][f][1] - mx[f][1]);
      const float p2 = mx[f][0] == -INFINITY ? 0.f : ex2_approx(sc[t][f][2] - mx[f][0]);
      const float p3 = mx[f][1] == -INFINITY ? 0.f : ex2_approx(sc[t][f][3] - mx[f][1]);
      l[f][0] += p0 + p2;
      l[f][1] += p1 + p3;
      pw[c0][16 * t + g8] = bits16<T>(p0);
      pw[c0 + 1][16 * t + g8] = bits16<T>(p1);
      pw[c0][16 * t + g8 + 8] = bits16<T>(p2);
      pw[c0 + 1][16 * t + g8 + 8] = bits16<T>(p3);
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[f][0] += __shfl_xor_sync(0xffffffffu, l[f][0], o);
      l[f][1] += __shfl_xor_sync(0xffffffffu, l[f][1], o);
    }
  }
  __syncwarp();

  // ---- output: dims 8(g8 + 8m) + 2i2 (+1) for columns 8f + 2q4, 8f + 2q4 + 1
  float o[NF][NM * 4][4];
#pragma unroll
  for (int f = 0; f < NF; ++f)
#pragma unroll
    for (int b = 0; b < NM * 4; ++b) o[f][b][0] = o[f][b][1] = o[f][b][2] = o[f][b][3] = 0.f;
#pragma unroll
  for (int t = 0; t < kDecTiles; ++t) {
    if (t < ntile) {
      if (t + 1 < ntile) load_v(t + 1, vb[(t + 1) & 1]);
      const uint4 (&vr)[4][NM] = vb[t & 1];
#pragma unroll
      for (int f = 0; f < NF; ++f) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&pw[kDecCols * f + g8][16 * t + 2 * q4]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&pw[kDecCols * f + g8][16 * t + 2 * q4 + 8]);
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            const uint32_t x0 = word(vr[0][m], i2), x1 = word(vr[1][m], i2);
            const uint32_t x2 = word(vr[2][m], i2), x3 = word(vr[3][m], i2);
            mma16816<T>(o[f][m * 4 + i2], __byte_perm(x0, x1, 0x5410), __byte_perm(x0, x1, 0x7632),
                        __byte_perm(x2, x3, 0x5410), __byte_perm(x2, x3, 0x7632), b0, b1);
          }
      }
    }
  }
  // The warp's partial: columns 8f + 2q4, 8f + 2q4 + 1 (those of the k rows), rows of dims.
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const int c0 = kDecCols * f + 2 * q4;
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const int d0 = 8 * (g8 + 8 * m) + 2 * i2;
        if (c0 < ncols)
          *reinterpret_cast<float2*>(&sO[warp][c0][d0]) = make_float2(o[f][m * 4 + i2][0], o[f][m * 4 + i2][2]);
        if (c0 + 1 < ncols)
          *reinterpret_cast<float2*>(&sO[warp][c0 + 1][d0]) = make_float2(o[f][m * 4 + i2][1], o[f][m * 4 + i2][3]);
      }
    if (g8 == 0) {
      sM[warp][c0] = mx[f][0];
      sL[warp][c0] = l[f][0];
      sM[warp][c0 + 1] = mx[f][1];
      sL[warp][c0 + 1] = l[f][1];
    }
  }
  __syncthreads();

  // ---- the split's partial: the warps' partials merged in warp order.  Partial
  // row (s * k + r, query head gk * G + h) for column (r, h).
  auto part_row = [&](int c) { return ((long long)(s * kr + c / G) * a.hq + gk * G + c % G) * a.max_splits; };
  for (int i = threadIdx.x; i < ncols * D; i += kDecWarps * 32) {
    const int h = i / D, dd = i % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, sM[w][h]);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (sM[w][h] != -INFINITY) v += ex2_approx(sM[w][h] - m) * sO[w][h][dd];
    a.part_o[(part_row(h) + split) * D + dd] = v;
  }
  if (threadIdx.x < ncols) {
    const int h = threadIdx.x;
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, sM[w][h]);
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (sM[w][h] != -INFINITY) l += ex2_approx(sM[w][h] - m) * sL[w][h];
    const long long idx = part_row(h) + split;
    a.part_ml[idx * 2 + 0] = m;
    a.part_ml[idx * 2 + 1] = l;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const AttnArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int kr = a.dec_rows;
  const int s = blockIdx.x / kr, r = blockIdx.x % kr, h = blockIdx.y, dd = threadIdx.x;
  if (seq_rows(a.rows, s) != kr) return;
  const int past = a.past[s];
  if (past < 0 || past + kr > a.max_ctx) return;
  const int n = past + r + 1;  // the keys row r sees
  const int nsplit = (n + kDecodeSplit - 1) / kDecodeSplit;
  const long long base = ((long long)(s * kr + r) * a.hq + h) * a.max_splits;
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
  out[((long long)(seq_row0(a.rows, s) + r) * a.hq + h) * D + dd] = from_float<T>(o);
}

template <typename T, int D>
cudaError_t launch_decode_t(const AttnArgs& a, cudaStream_t st) {
  if ((long long)a.rows.num_seqs * a.max_splits >= (1ll << 31) || a.hkv > 65535 ||
      (long long)a.rows.num_seqs * a.dec_rows >= (1ll << 31) || a.dec_rows < 1 ||
      a.dec_rows * a.group > kDecCols * 2)
    return cudaErrorInvalidValue;
  const dim3 grid(a.rows.num_seqs * a.max_splits, a.hkv);
  cudaError_t e = a.dec_rows == 1 ? launch_pdl(decode_split_kernel<T, D>, grid, dim3(kDecWarps * 32), 0, st, a)
                  : a.dec_rows * a.group <= kDecCols
                      ? launch_pdl(decode_rows_kernel<T, D, 1>, grid, dim3(kDecWarps * 32), 0, st, a)
                      : launch_pdl(decode_rows_kernel<T, D, 2>, grid, dim3(kDecWarps * 32), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_combine_kernel<T, D>, dim3(a.rows.num_seqs * a.dec_rows, a.hq), dim3(D), 0, st, a);
}

}  // namespace

bool decode_supported(int d, int group, int dtype) {
  return (d == 64 || d == 128) && (group == 1 || group == 2 || group == 4 || group == 8) &&
         (dtype == CP_BF16 || dtype == CP_F16);
}

cudaError_t launch_decode(const AttnArgs& a, int dtype, cudaStream_t st) {
  if (a.rows.num_seqs == 0 || a.max_splits == 0) return cudaSuccess;
  if (dtype == CP_BF16) return a.d == 64 ? launch_decode_t<__nv_bfloat16, 64>(a, st)
                                         : launch_decode_t<__nv_bfloat16, 128>(a, st);
  return a.d == 64 ? launch_decode_t<__half, 64>(a, st) : launch_decode_t<__half, 128>(a, st);
}

}  // namespace cp
