// attn_f32.cu -- chunk attention in fp32 on the CUDA cores (SIMT FFMA).
//
// The fp32 path exists for the 1e-4 accuracy class of the one-layer example
// (Ultralytics glossary "Chunked Prefill", "How chunked prefill works": 8 heads
// x 64 dims, fp32).  TF32 tensor-core products would not meet that bound, so
// this kernel multiplies in full fp32.  Its roofline is the FP32 FMA rate.
//
// A CTA owns 16 consecutive query rows of one query head and splits their key
// walk over kSplits warp groups (4 for D = 64, 2 for D = 128): group `sp` takes
// the 32-key tiles sp, sp + kSplits, ...  The example's chunks hold only 2048
// query rows in all, so the split is what puts several warps on each SM
// sub-partition.  Within a group, warp w owns rows 4w .. 4w+3 outright (scores,
// online softmax state and output).  Each group streams its tiles through its
// own two-stage shared-memory ring with cp.async (16-byte copies, zero-filled
// past the keys), one tile ahead.  Per tile and warp:
//   scores  lane l computes key l of its 4 rows from a float4 of each Q row (a
//           broadcast) and of its K row per 4 dimensions;
//   softmax online, in the log2 domain: the row max by a warp reduction, the
//           row sum kept per lane and reduced once at the end;
//   output  P goes to the warp's rows of its group's P tile, and lane l
//           accumulates D/32 consecutive output dimensions of its 4 rows from a
//           float4 of P (4 keys, a broadcast) and vectors of V rows.
// At the end the groups' partial results (max, sum, output) meet in shared
// memory and are merged in group order.  Every dot product runs over
// dimensions in ascending order, and every output sum over a group's keys in
// ascending order, so the result depends only on the inputs.  Works on all
// three cache layouts through cp_kv.cuh.
//
// One-call chunk on a contiguous cache (`fused`): the keys at or past the
// cached length are this call's rows, read from k_new / v_new; the CTAs of the
// first query head of each KV group copy their 16 rows' K and V into the
// cache (no CTA of the launch reads those slots from the cache), and the last
// CTA to take a ticket, after every CTA has read the lengths, advances them
// ([Wiki] 一.1 and 四).
#include <atomic>
#include <cmath>
#include <cstdint>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kRows = 16;     // query rows per CTA
constexpr int kKeys = 32;     // keys per tile
constexpr int kRowWarps = 4;  // warps per group; warp w owns rows 4w .. 4w+3

template <int D>
struct F32Cfg {
  static constexpr int kSplits = D == 64 ? 4 : 2;  // warp groups splitting the key walk
  static constexpr int kThreads = kSplits * kRowWarps * 32;
  static constexpr int KS = D + 4;  // K row stride in floats: float4 reads by 8 lanes hit 8 distinct 16-byte slots
};

template <int D>
struct F32Smem {
  static constexpr int S = F32Cfg<D>::kSplits;
  float q[kRows][D];
  union {
    struct {
      float k[S][2][kKeys][F32Cfg<D>::KS];
      float v[S][2][kKeys][D];
    } ring;
    struct {  // the groups' partial results, after the walk
      float o[S][kRows][D];
      float m[S][kRows];
      float l[S][kRows];
    } part;
  };
  float p[S][kRows][kKeys];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = fill ? 16 : 0;  // 0: the 16 bytes are zero-filled and src is not read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A named barrier for the 128 threads of warp group `sp` (ids 1 .. kSplits;
// 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int sp) {
  asm volatile("bar.sync %0, %1;" ::"r"(sp + 1), "n"(kRowWarps * 32) : "memory");
}

// The ticket of a one-call chunk: every CTA takes one after all its threads
// have read the lengths; the last one advances them by commit_add and resets
// the counter.  A counter found above the grid size was not zero before the
// launch: reported as CP_DEV_BOUNDS.
__device__ __forceinline__ void take_ticket(const AttnArgs& a) {
  __threadfence();
  const unsigned total = gridDim.x * gridDim.y * gridDim.z;
  const unsigned t = atomicAdd(a.ticket, 1u);
  if (t == total - 1) {
    __threadfence();
    for (int i = 0; i < a.rows.num_seqs; ++i) a.commit_lens[i] += a.commit_add;
    __threadfence();
    atomicExch(a.ticket, 0u);
  } else if (t >= total && a.status) {
    atomicOr(a.status, CP_DEV_BOUNDS);
  }
}

template <int D>
__global__ void __launch_bounds__(F32Cfg<D>::kThreads) attn_f32_kernel(const AttnArgs a) {
  using C = F32Cfg<D>;
  constexpr int S = C::kSplits;
  constexpr int DV = D / 32;  // output dimensions per lane
  extern __shared__ __align__(16) uint8_t f32_smem_raw[];
  F32Smem<D>& sm = *reinterpret_cast<F32Smem<D>*>(f32_smem_raw);

  pdl_launch_dependents();
  pdl_wait();
  // The length advance of a one-call chunk with a separate append: `past` is
  // then a copy of the lengths, so CTA (0, 0, 0) may advance them at once.
  if (a.commit_lens && !a.ticket && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    for (int i = threadIdx.x; i < a.rows.num_seqs; i += C::kThreads) a.commit_lens[i] += a.commit_add;
  const int s = blockIdx.z;
  const int h = blockIdx.y;
  const int g = h / a.group;
  const int rows = seq_rows(a.rows, s);
  const int t0 = blockIdx.x * kRows;
  bool work = t0 < rows && rows >= a.min_rows;
  int past = 0;
  if (work) {
    past = a.past[s];
    if (past < 0 || past + rows > a.max_ctx) {
      if (a.status && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
      work = false;
    }
  }
  if (a.ticket) {
    __syncthreads();  // every thread has read its length before this CTA takes a ticket
    if (threadIdx.x == 0) take_ticket(a);
  }
  if (!work) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp / kRowWarps;                   // this warp's group
  const int rw = warp % kRowWarps;                   // its rows: 4 rw .. 4 rw + 3
  const int gtid = threadIdx.x % (kRowWarps * 32);  // thread index within the group
  const int n = past + rows;
  const int t_last = min(t0 + kRows, rows) - 1;
  const SeqKeys keys = seq_keys(a, s, n, past + t_last);
  const long long row0 = seq_row0(a.rows, s);

  const float* q = static_cast<const float*>(a.q);
  const float* kc = static_cast<const float*>(a.k);
  const float* vc = static_cast<const float*>(a.v);
  const float* kn = static_cast<const float*>(a.k_new);
  const float* vn = static_cast<const float*>(a.v_new);
  const bool fused = a.fused != 0;

  // K/V tile `tile` (keys 32 tile ..) into this group's stage `st`, by the
  // group's threads: 16-byte chunks, keys past the walk (or on an
  // out-of-range page) zero-filled.
  auto load_tile = [&](int tile, int st) {
    constexpr int kChunks = D / 4;  // 16-byte chunks per row
    for (int c = gtid; c < kKeys * kChunks; c += kRowWarps * 32) {
      const int r = c / kChunks, c4 = c % kChunks;
      const int j = tile * kKeys + r;
      const bool from_new = fused && j >= past;  // this call's row j - past of sequence s
      long long off = -1;
      if (j < keys.nkeys) {
        off = from_new ? (((long long)s * rows + (j - past)) * a.hkv + g) * D : key_offset(a.cache, a.hkv, D, s, g, j);
        if (off < 0 && a.status && c4 == 0) atomicOr(a.status, CP_DEV_BOUNDS);
      }
      const bool ok = off >= 0;
      const long long e = ok ? off + 4 * c4 : 0;
      cp_async16(&sm.ring.k[sp][st][r][4 * c4], (from_new ? kn : kc) + e, ok);
      cp_async16(&sm.ring.v[sp][st][r][4 * c4], (from_new ? vn : vc) + e, ok);
    }
  };

  if (fused && h % a.group == 0) {
    // This CTA's rows of KV head g into their cache slots, 16 bytes at a time.
    float* kdst = static_cast<float*>(a.k_cache);
    float* vdst = static_cast<float*>(a.v_cache);
    for (int e = threadIdx.x; e < kRows * (D / 4); e += C::kThreads) {
      const int r = e / (D / 4), c4 = e % (D / 4);
      const int t = t0 + r;
      if (t >= rows) continue;
      const long long src = (((long long)s * rows + t) * a.hkv + g) * D + 4 * c4;
      const long long dst = (((long long)s * a.hkv + g) * a.cache.capacity + past + t) * D + 4 * c4;
      *reinterpret_cast<float4*>(kdst + dst) = *reinterpret_cast<const float4*>(kn + src);
      *reinterpret_cast<float4*>(vdst + dst) = *reinterpret_cast<const float4*>(vn + src);
    }
  }

  const int ntiles = (keys.nkeys + kKeys - 1) / kKeys;
  const int nmine = ntiles > sp ? (ntiles - sp + S - 1) / S : 0;  // this group's tiles: sp + S i
  if (nmine > 0) load_tile(sp, 0);
  cp_async_commit();
  for (int e = threadIdx.x; e < kRows * D; e += C::kThreads) {
    const int r = e / D, d = e % D;
    const int t = t0 + r;
    sm.q[r][d] = t < rows ? q[((row0 + t) * a.hq + h) * D + d] : 0.f;
  }
  __syncthreads();  // Q is in shared memory for every group

  int p_row[4];
  float m[4], l[4], o[4][DV];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * rw + i;
    p_row[i] = t < rows ? past + t : -1;  // absolute position; -1: no row (sees nothing)
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int u = 0; u < DV; ++u) o[i][u] = 0.f;
  }

  for (int it = 0; it < nmine; ++it) {
    const int st = it & 1;
    const int tile = sp + S * it;
    if (it + 1 < nmine) {
      load_tile(tile + S, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    group_sync(sp);  // the group's tile is in shared memory for all its warps

    // ---- scores of key 32 tile + lane for rows 4 rw .. 4 rw + 3
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 kv = *reinterpret_cast<const float4*>(&sm.ring.k[sp][st][lane][4 * d4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[4 * rw + i][4 * d4]);
        sc[i] = fmaf(qv.x, kv.x, sc[i]);
        sc[i] = fmaf(qv.y, kv.y, sc[i]);
        sc[i] = fmaf(qv.z, kv.z, sc[i]);
        sc[i] = fmaf(qv.w, kv.w, sc[i]);
      }
    }
    // ---- visibility and the online softmax, row by row
    const int j = tile * kKeys + lane;
    const bool in = j < keys.nkeys;
    const int pos = in ? key_pos(a.cache, keys, j) : 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool vis = in && pos <= p_row[i] && pos >= keys.lo;
      const float x = vis ? sc[i] * a.scale_log2 : -INFINITY;
      float mt = x;
#pragma unroll
      for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m[i], mt);
      float pr = 0.f;
      if (m_new != -INFINITY) {  // else nothing visible yet: the row's state stays as it is
        const float alpha = (m[i] == -INFINITY) ? 0.f : ex2_approx(m[i] - m_new);
        pr = x == -INFINITY ? 0.f : ex2_approx(x - m_new);
        l[i] = l[i] * alpha + pr;
        m[i] = m_new;
#pragma unroll
        for (int u = 0; u < DV; ++u) o[i][u] *= alpha;
      }
      sm.p[sp][4 * rw + i][lane] = pr;
    }
    __syncwarp();  // the warp's own rows of P are written (no other warp reads them)

    // ---- O[rows][lane * DV ..] += P V over the tile's keys in ascending order
#pragma unroll 2
    for (int k4 = 0; k4 < kKeys / 4; ++k4) {
      float4 pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(&sm.p[sp][4 * rw + i][4 * k4]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float vv[DV];
        if constexpr (DV == 4) {
          const float4 t = *reinterpret_cast<const float4*>(&sm.ring.v[sp][st][4 * k4 + kk][4 * lane]);
          vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(&sm.ring.v[sp][st][4 * k4 + kk][2 * lane]);
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
    group_sync(sp);  // the group is done with stage `st` before its next loads overwrite it
  }
  cp_async_wait<0>();  // no copy into shared memory outlives the walk
  __syncthreads();     // every group is done with the ring: it now holds the partial results

  // ---- the groups' partials, then their merge in group order
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lt = l[i];
#pragma unroll
    for (int off = 16; off; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    const int r = 4 * rw + i;
    if (lane == 0) {
      sm.part.m[sp][r] = m[i];
      sm.part.l[sp][r] = lt;
    }
#pragma unroll
    for (int u = 0; u < DV; ++u) sm.part.o[sp][r][DV * lane + u] = o[i][u];
  }
  __syncthreads();
  float* out = static_cast<float*>(a.out);
  for (int e = threadIdx.x; e < kRows * D; e += C::kThreads) {
    const int r = e / D, d = e % D;
    const int t = t0 + r;
    if (t >= rows) continue;
    float mm = -INFINITY;
#pragma unroll
    for (int k = 0; k < S; ++k) mm = fmaxf(mm, sm.part.m[k][r]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int k = 0; k < S; ++k) {
      const float mk = sm.part.m[k][r];
      const float w = mk == -INFINITY ? 0.f : ex2_approx(mk - mm);
      acc = fmaf(w, sm.part.o[k][r][d], acc);
      lsum = fmaf(w, sm.part.l[k][r], lsum);
    }
    out[((row0 + t) * a.hq + h) * D + d] = lsum > 0.f ? acc * (1.f / lsum) : 0.f;
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
  return launch_pdl(attn_f32_kernel<D>, grid, dim3(F32Cfg<D>::kThreads), (size_t)smem, st, a);
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a, int rows_bound, cudaStream_t st) {
  dim3 grid((rows_bound + kRows - 1) / kRows, a.hq, a.rows.num_seqs);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  if (a.d == 64) return launch_f32_t<64>(a, grid, st);
  return launch_f32_t<128>(a, grid, st);
}

}  // namespace cp
