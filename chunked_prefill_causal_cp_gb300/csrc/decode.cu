// decode.cu -- single-row (decode) attention on the memory-bound split-KV path.
//
// A decode row reads its sequence's whole K/V once and does ~1 FLOP per byte
// (Ultralytics glossary "Chunked Prefill", "Prefill, decode and generation
// stalls": decode is memory-bandwidth bound), so this path is built around
// coalesced 16-byte loads, not the tensor cores.
//
// decode_split_kernel: one CTA per (split of 512 keys, KV head, sequence).
//   The GQA group's query heads share every K/V row the CTA loads.  A group
//   of D/8 lanes holds one key row (8 elements = 16 bytes per lane); each
//   lane keeps the group's q values for its 8 dimensions, the partial dot
//   products are reduced with xor shuffles, scores go to shared memory, the
//   CTA takes the split's max and sum (log2 domain), then streams V once
//   and writes the unnormalised partial output.
// decode_combine_kernel: merges a row's split partials in split order
//   (log-sum-exp), so the result depends only on the row's own context.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kDecWarps = 4;
constexpr int kDecUnroll = 4;

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& raw, float (&f)[8]) {
  const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = static_cast<float>(e[i]);
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecWarps * 32) decode_split_kernel(const AttnArgs a) {
  constexpr int LPK = D / 8;          // lanes per key row
  constexpr int KPW = 32 / LPK;       // key rows per warp per step
  constexpr int KPS = kDecWarps * KPW;  // key rows per CTA per step
  __shared__ float sc[G][kDecodeSplit];
  __shared__ float red[kDecWarps][G][D];
  __shared__ float s_m[G], s_l[G];

  const int split = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  if (seq_rows(a.rows, s) != 1) return;
  const int past = a.past[s];
  const int n = past + 1;
  if (past < 0 || n > a.max_ctx) {
    if (a.status && threadIdx.x == 0 && split == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int k0 = split * kDecodeSplit;
  if (k0 >= n) return;
  const int nk = min(n - k0, kDecodeSplit);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane % LPK;          // which 8-element slice of the row
  const int kslot = warp * KPW + lane / LPK;
  const long long qrow = (long long)seq_row0(a.rows, s) * a.hq;

  float qv[G][8];
  {
    const T* q = static_cast<const T*>(a.q);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 raw = *reinterpret_cast<const uint4*>(q + (qrow + g * G + h) * D + sub * 8);
      unpack8<T>(raw, qv[h]);
#pragma unroll
      for (int e = 0; e < 8; ++e) qv[h][e] *= a.scale_log2;
    }
  }
  const T* kc = static_cast<const T*>(a.k);
  const T* vc = static_cast<const T*>(a.v);

  // ---- scores
  for (int base = 0; base < nk; base += KPS * kDecUnroll) {
    uint4 raw[kDecUnroll];
    bool ok[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int kk = base + u * KPS + kslot;
      ok[u] = false;
      raw[u] = make_uint4(0, 0, 0, 0);
      if (kk < nk) {
        const long long off = key_offset(a.cache, a.hkv, D, s, g, k0 + kk);
        if (off >= 0) {
          raw[u] = __ldg(reinterpret_cast<const uint4*>(kc + off + sub * 8));
          ok[u] = true;
        } else if (a.status) {
          atomicOr(a.status, CP_DEV_BOUNDS);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      float kf[8];
      unpack8<T>(raw[u], kf);
      float dot[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qv[h][e], kf[e], acc);
#pragma unroll
        for (int off = LPK / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        dot[h] = acc;
      }
      const int kk = base + u * KPS + kslot;
      if (sub == 0 && kk < nk) {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h][kk] = ok[u] ? dot[h] : -INFINITY;
      }
    }
  }
  __syncthreads();

  // ---- split max / sum per query head (log2 domain)
  for (int h = warp; h < G; h += kDecWarps) {
    float m = -INFINITY;
    for (int kk = lane; kk < nk; kk += 32) m = fmaxf(m, sc[h][kk]);
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int kk = lane; kk < nk; kk += 32) {
      const float p = (m == -INFINITY) ? 0.f : ex2_approx(sc[h][kk] - m);
      sc[h][kk] = p;
      l += p;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) {
      s_m[h] = m;
      s_l[h] = l;
    }
  }
  __syncthreads();

  // ---- p . V
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
  for (int base = 0; base < nk; base += KPS * kDecUnroll) {
    uint4 raw[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int kk = base + u * KPS + kslot;
      raw[u] = make_uint4(0, 0, 0, 0);
      if (kk < nk) {
        const long long off = key_offset(a.cache, a.hkv, D, s, g, k0 + kk);
        if (off >= 0) raw[u] = __ldg(reinterpret_cast<const uint4*>(vc + off + sub * 8));
      }
    }
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int kk = base + u * KPS + kslot;
      if (kk < nk) {
        float vf[8];
        unpack8<T>(raw[u], vf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = sc[h][kk];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(p, vf[e], acc[h][e]);
        }
      }
    }
  }
  // Sum the KPW key slots of the warp (lanes with the same `sub`).
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int off = LPK; off < 32; off <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
  if (lane < LPK) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) red[warp][h][sub * 8 + e] = acc[h][e];
  }
  __syncthreads();
  const long long part_base = ((long long)s * a.hq + g * G) * a.max_splits;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, dd = i % D;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) v += red[w][h][dd];
    a.part_o[((part_base + (long long)h * a.max_splits) + split) * D + dd] = v;
  }
  if (threadIdx.x < G) {
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

template <typename T, int D, int G>
cudaError_t launch_decode_t(const AttnArgs& a, cudaStream_t st) {
  dim3 grid(a.max_splits, a.hkv, a.rows.num_seqs);
  decode_split_kernel<T, D, G><<<grid, kDecWarps * 32, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<T, D><<<dim3(a.rows.num_seqs, a.hq), D, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_d(const AttnArgs& a, cudaStream_t st) {
  switch (a.group) {
    case 1: return launch_decode_t<T, D, 1>(a, st);
    case 2: return launch_decode_t<T, D, 2>(a, st);
    case 4: return launch_decode_t<T, D, 4>(a, st);
    case 8: return launch_decode_t<T, D, 8>(a, st);
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
