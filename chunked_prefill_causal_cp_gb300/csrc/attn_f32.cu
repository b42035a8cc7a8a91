// attn_f32.cu -- chunk attention in fp32 on the CUDA cores (SIMT FFMA).
//
// The fp32 path exists for the 1e-4 accuracy class of the one-layer example
// (Ultralytics glossary "Chunked Prefill", "How chunked prefill works": 8 heads
// x 64 dims, fp32).  TF32 tensor-core products would not meet that bound, so
// this kernel multiplies in full fp32.  Its roofline is the FP32 FMA rate.
//
// A CTA of 4 warps owns 16 consecutive query rows of one query head; warp w
// owns rows 4w .. 4w+3 outright (their scores, softmax state and output), so
// only the K/V tiles are shared across warps.  (Two rows per warp in 8 warps,
// or one in 16, measured slower: the extra warps do not hide more latency
// than the lost register reuse costs in instructions.)  64-key K/V tiles stream through
// a two-stage shared-memory ring with cp.async (16-byte copies, zero-filled
// past the keys), one tile ahead of the arithmetic.  Per tile and warp:
//   scores  lane l computes keys l and l + 32 of its 4 rows: a float4 of each
//           row of Q (a broadcast) and of each of its two K rows per 4 dims;
//   softmax online, in the log2 domain: the row max by a warp reduction, the
//           row sum kept per lane and reduced once at the end;
//   output  P goes to the warp's rows of a shared tile, and lane l
//           accumulates D/32 consecutive output dimensions of its 4 rows from
//           a float4 of P (4 keys, a broadcast) and V rows read as vectors.
// Every dot product runs over dimensions, and every output sum over keys, in
// ascending order.  Works on all three cache layouts through cp_kv.cuh.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kRows = 16;     // query rows per CTA
constexpr int kKeys = 64;     // keys per tile
constexpr int kWarps = 4;     // warps per CTA; warp w owns rows 4w .. 4w+3
constexpr int kThreads = kWarps * 32;
static_assert(kRows == 4 * kWarps, "each warp owns four rows");

template <int D>
struct F32Smem {
  static constexpr int KS = D + 4;  // K row stride in floats: float4 reads by 8 lanes hit 8 distinct 16-byte slots
  float q[kRows][D];
  float k[2][kKeys][KS];
  float v[2][kKeys][D];
  float p[kRows][kKeys];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = fill ? 16 : 0;  // 0: the 16 bytes are zero-filled and src is not read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D>
__global__ void __launch_bounds__(kThreads) attn_f32_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) uint8_t f32_smem_raw[];
  F32Smem<D>& sm = *reinterpret_cast<F32Smem<D>*>(f32_smem_raw);
  constexpr int DV = D / 32;  // output dimensions per lane

  pdl_launch_dependents();
  pdl_wait();
  const int s = blockIdx.z;
  const int h = blockIdx.y;
  const int g = h / a.group;
  const int rows = seq_rows(a.rows, s);
  const int t0 = blockIdx.x * kRows;
  if (t0 >= rows || rows < a.min_rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int past = a.past[s];
  const int n = past + rows;
  if (n > a.max_ctx || past < 0) {
    if (a.status && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int t_last = min(t0 + kRows, rows) - 1;
  const SeqKeys keys = seq_keys(a, s, n, past + t_last);
  const long long row0 = seq_row0(a.rows, s);

  const float* q = static_cast<const float*>(a.q);
  const float* kc = static_cast<const float*>(a.k);
  const float* vc = static_cast<const float*>(a.v);

  // K/V tile j0 .. j0+63 into stage `st`: 16-byte chunks, keys past the walk
  // (or on an out-of-range page) zero-filled.
  auto load_tile = [&](int j0, int st) {
    constexpr int kChunks = D / 4;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < kKeys * kChunks; c += kThreads) {
      const int r = c / kChunks, c4 = c % kChunks;
      const int j = j0 + r;
      long long off = -1;
      if (j < keys.nkeys) {
        off = key_offset(a.cache, a.hkv, D, s, g, j);
        if (off < 0 && a.status && c4 == 0) atomicOr(a.status, CP_DEV_BOUNDS);
      }
      const bool ok = off >= 0;
      const long long e = ok ? off + 4 * c4 : 0;
      cp_async16(&sm.k[st][r][4 * c4], kc + e, ok);
      cp_async16(&sm.v[st][r][4 * c4], vc + e, ok);
    }
  };

  load_tile(0, 0);
  cp_async_commit();
  for (int e = threadIdx.x; e < kRows * D; e += kThreads) {
    const int r = e / D, d = e % D;
    const int t = t0 + r;
    sm.q[r][d] = t < rows ? q[((row0 + t) * a.hq + h) * D + d] : 0.f;
  }

  int p_row[4];
  float m[4], l[4], o[4][DV];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * warp + i;
    p_row[i] = t < rows ? past + t : -1;  // absolute position; -1: no row (sees nothing)
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int u = 0; u < DV; ++u) o[i][u] = 0.f;
  }

  const int ntiles = (keys.nkeys + kKeys - 1) / kKeys;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int st = tile & 1;
    if (tile + 1 < ntiles) {
      load_tile((tile + 1) * kKeys, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile `tile` (and, the first time, Q) is in shared memory for every warp

    // ---- scores of keys j0 + lane and j0 + lane + 32 for rows 4w .. 4w+3
    const int j0 = tile * kKeys;
    float sc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i][0] = sc[i][1] = 0.f;
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 k0 = *reinterpret_cast<const float4*>(&sm.k[st][lane][4 * d4]);
      const float4 k1 = *reinterpret_cast<const float4*>(&sm.k[st][lane + 32][4 * d4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[4 * warp + i][4 * d4]);
        sc[i][0] = fmaf(qv.x, k0.x, sc[i][0]);
        sc[i][0] = fmaf(qv.y, k0.y, sc[i][0]);
        sc[i][0] = fmaf(qv.z, k0.z, sc[i][0]);
        sc[i][0] = fmaf(qv.w, k0.w, sc[i][0]);
        sc[i][1] = fmaf(qv.x, k1.x, sc[i][1]);
        sc[i][1] = fmaf(qv.y, k1.y, sc[i][1]);
        sc[i][1] = fmaf(qv.z, k1.z, sc[i][1]);
        sc[i][1] = fmaf(qv.w, k1.w, sc[i][1]);
      }
    }
    // ---- visibility and the online softmax, row by row
    int pos[2];
    bool in[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = j0 + lane + 32 * c;
      in[c] = j < keys.nkeys;
      pos[c] = in[c] ? key_pos(a.cache, keys, j) : 0;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const bool vis = in[c] && pos[c] <= p_row[i] && pos[c] >= keys.lo;
        x[c] = vis ? sc[i][c] * a.scale_log2 : -INFINITY;
      }
      float mt = fmaxf(x[0], x[1]);
#pragma unroll
      for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m[i], mt);
      float p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {  // else nothing visible yet: the row's state stays as it is
        const float alpha = (m[i] == -INFINITY) ? 0.f : ex2_approx(m[i] - m_new);
        p0 = x[0] == -INFINITY ? 0.f : ex2_approx(x[0] - m_new);
        p1 = x[1] == -INFINITY ? 0.f : ex2_approx(x[1] - m_new);
        l[i] = l[i] * alpha + (p0 + p1);
        m[i] = m_new;
#pragma unroll
        for (int u = 0; u < DV; ++u) o[i][u] *= alpha;
      }
      sm.p[4 * warp + i][lane] = p0;
      sm.p[4 * warp + i][lane + 32] = p1;
    }
    __syncwarp();  // the warp's own rows of P are written (no other warp reads them)

    // ---- O[rows][lane * DV ..] += P V, keys in ascending order
#pragma unroll 2
    for (int k4 = 0; k4 < kKeys / 4; ++k4) {
      float4 pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(&sm.p[4 * warp + i][4 * k4]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float vv[DV];
        if constexpr (DV == 4) {
          const float4 t = *reinterpret_cast<const float4*>(&sm.v[st][4 * k4 + kk][4 * lane]);
          vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(&sm.v[st][4 * k4 + kk][2 * lane]);
          vv[0] = t.x; vv[1] = t.y;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pk = kk == 0 ? pv[i].x : kk == 1 ? pv[i].y : kk == 2 ? pv[i].z : pv[i].w;
#pragma unroll
          for (int u = 0; u < DV; ++u) o[i][u] = fmaf(pk, vv[u], o[i][u]);
        }
      }
    }
    __syncthreads();  // every warp is done with stage `st` before the next loads overwrite it
  }
  cp_async_wait<0>();  // no copy into shared memory outlives the loop

  float* out = static_cast<float*>(a.out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lt = l[i];
#pragma unroll
    for (int off = 16; off; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    const int t = t0 + 4 * warp + i;
    if (t >= rows) continue;
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    float* dst = out + ((row0 + t) * a.hq + h) * D + DV * lane;
#pragma unroll
    for (int u = 0; u < DV; ++u) dst[u] = o[i][u] * inv;
  }
}

template <int D>
cudaError_t launch_f32_t(const AttnArgs& a, dim3 grid, cudaStream_t st) {
  const int smem = (int)sizeof(F32Smem<D>);
  // The dynamic shared-memory limit is a per-device function attribute: raise
  // it once per device, so later calls (also under stream capture) only launch.
  static std::atomic<uint64_t> ready_mask{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(ready_mask.load() & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ready_mask.fetch_or(bit);
  }
  return launch_pdl(attn_f32_kernel<D>, grid, dim3(kThreads), (size_t)smem, st, a);
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a, int rows_bound, cudaStream_t st) {
  dim3 grid((rows_bound + kRows - 1) / kRows, a.hq, a.rows.num_seqs);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  if (a.d == 64) return launch_f32_t<64>(a, grid, st);
  return launch_f32_t<128>(a, grid, st);
}

}  // namespace cp
