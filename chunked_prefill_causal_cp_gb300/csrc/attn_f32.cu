// attn_f32.cu -- chunk attention in fp32 on the CUDA cores (SIMT FFMA).
//
// The fp32 path exists for the 1e-4 accuracy class of the one-layer example
// (Ultralytics glossary "Chunked Prefill", "How chunked prefill works": 8 heads
// x 64 dims, fp32).  TF32 tensor-core products would not meet that bound, so
// this kernel multiplies in full fp32.
//
// One warp owns one query row; a CTA holds 8 consecutive rows of one query
// head and stages 32-key K/V tiles in shared memory.  Lane j scores key j of
// the tile, the warp keeps an online softmax (running max / sum in the log2
// domain) and each lane accumulates D/32 output dimensions.  Works on all
// three cache layouts through cp_kv.cuh.
#include <cmath>
#include <cstdint>

#include "cp_internal.h"
#include "cp_kv.cuh"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kKeysPerTile = 32;

template <int D>
__global__ void __launch_bounds__(256) attn_f32_kernel(const AttnArgs a) {
  __shared__ float ks[kKeysPerTile][D + 1];
  __shared__ float vs[kKeysPerTile][D];
  __shared__ float qs[kRowsPerCta][D];

  pdl_launch_dependents();
  pdl_wait();
  const int s = blockIdx.z;
  const int h = blockIdx.y;
  const int g = h / a.group;
  const int rows = seq_rows(a.rows, s);
  const int t0 = blockIdx.x * kRowsPerCta;
  if (t0 >= rows || rows < a.min_rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int past = a.past[s];
  const int n = past + rows;
  if (n > a.max_ctx || past < 0) {
    if (a.status && threadIdx.x == 0) atomicOr(a.status, CP_DEV_BOUNDS);
    return;
  }
  const int t_last = min(t0 + kRowsPerCta, rows) - 1;
  const SeqKeys keys = seq_keys(a, s, n, past + t_last);
  const int my_t = t0 + warp;
  const bool row_ok = my_t < rows;
  const int my_p = past + my_t;
  const long long qrow = (long long)(seq_row0(a.rows, s) + my_t) * a.hq + h;

  const float* q = static_cast<const float*>(a.q);
  const float* kc = static_cast<const float*>(a.k);
  const float* vc = static_cast<const float*>(a.v);
  for (int d = lane; d < D; d += 32) qs[warp][d] = row_ok ? q[qrow * D + d] : 0.f;

  float m = -INFINITY, l = 0.f;
  float o[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) o[i] = 0.f;

  for (int j0 = 0; j0 < keys.nkeys; j0 += kKeysPerTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeysPerTile * D; e += blockDim.x) {
      const int r = e / D, d = e % D;
      const int j = j0 + r;
      float kv = 0.f, vv = 0.f;
      if (j < keys.nkeys) {
        const long long off = key_offset(a.cache, a.hkv, D, s, g, j);
        if (off >= 0) {
          kv = kc[off + d];
          vv = vc[off + d];
        } else if (a.status && d == 0) {
          atomicOr(a.status, CP_DEV_BOUNDS);
        }
      }
      ks[r][d] = kv;
      vs[r][d] = vv;
    }
    __syncthreads();
    if (!row_ok) continue;
    const int j = j0 + lane;
    bool vis = false;
    if (j < keys.nkeys) {
      const int pos = key_pos(a.cache, keys, j);
      vis = pos <= my_p && pos >= keys.lo;
    }
    float sc = 0.f;
#pragma unroll 16
    for (int d = 0; d < D; ++d) sc = fmaf(qs[warp][d], ks[lane][d], sc);
    sc = vis ? sc * a.scale_log2 : -INFINITY;
    float tmax = sc;
#pragma unroll
    for (int off = 16; off; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);
    if (m_new == -INFINITY) continue;  // nothing visible yet
    const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
    const float p = vis ? ex2_approx(sc - m_new) : 0.f;
    float psum = p;
#pragma unroll
    for (int off = 16; off; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) o[i] *= alpha;
#pragma unroll 8
    for (int jj = 0; jj < kKeysPerTile; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) o[i] = fmaf(pj, vs[jj][lane + 32 * i], o[i]);
    }
  }
  if (!row_ok) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* out = static_cast<float*>(a.out);
#pragma unroll
  for (int i = 0; i < D / 32; ++i) out[qrow * D + lane + 32 * i] = o[i] * inv;
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a, int rows_bound, cudaStream_t st) {
  dim3 grid((rows_bound + kRowsPerCta - 1) / kRowsPerCta, a.hq, a.rows.num_seqs);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  if (a.d == 64) return launch_pdl(attn_f32_kernel<64>, grid, dim3(256), 0, st, a);
  return launch_pdl(attn_f32_kernel<128>, grid, dim3(256), 0, st, a);
}

}  // namespace cp
