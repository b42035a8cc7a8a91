// cp_oracle.cpp -- plain C++ CPU oracle for chunked-prefill causal attention.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
// CPU-baseline / reference leg of bench.py may load or call this library
// (through oracle/cpp.py).  It shares no code, header or table with the CUDA
// library under chunked_prefill_causal_cp_gb300/, and includes none of it.
//
// Plain and slow, meant to be checked by eye: every value is a double, every
// sum runs in index order, and the only concurrency is std::thread over
// independent (query row, head) pairs, each computed start to finish by one
// thread.  The functions follow, step for step, the same passages as the
// numpy oracle in cp_oracle.py (same names, same readings):
//
//   [Wiki]      ONNX GenAI Wiki, "Chunked Prefill": §一.1 append-only cache;
//               §一.2 the causal mask hides the split; §一.3 capacity vs
//               seqlens_k; §二/§三 chunks of W and the remainder; §四 query
//               padding (pad rows repeat the last real token, output cut back,
//               length rewound); §六 the ladder's top tier is W.
//   [Horizon]   Horizon developer blog, "【大模型】Chunk Prefill——把一次算不动的事拆成多次":
//               §3 rolling cache (concatenate, drop the oldest c); §4 the
//               (c, C) right-aligned mask filled with -32768, added to scores.
//   [Glossary]  Ultralytics glossary, "Chunked Prefill": "How chunked prefill
//               works" (token-budget steps; the one-layer example);
//               "Related techniques" (PagedAttention).
//
// Readings where the pages are silent: softmax scale 1/sqrt(D); query head h
// reads KV head h / (Hq / Hkv); seqlens_k counts valid slots; pad rows copy
// the last real row; the rolling cache starts all-zero and its mask is added
// to the scores; the scheduler is first-come-first-served with no per-prompt
// cap, and a prompt that finished decodes from the next step on.
//
// Layouts (all row-major doubles): a sequence's tokens are [n, H, D]; a
// contiguous cache is [B, Hkv, cap, D]; a rolling cache is [H, C, D]; a page
// pool is [num_pages, Hkv, page, D].
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

int g_threads = 0;  // 0: std::thread::hardware_concurrency()

int thread_count() {
  if (g_threads > 0) return g_threads;
  const unsigned h = std::thread::hardware_concurrency();
  return h > 0 ? (int)h : 1;
}

// body(i) for every i in [0, n); thread w takes i = w, w + T, w + 2T, ...
template <class F>
void for_each_index(int64_t n, F body) {
  const int64_t t = std::min<int64_t>(thread_count(), n);
  if (t <= 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int64_t w = 0; w < t; ++w)
    pool.emplace_back([&body, w, t, n] {
      for (int64_t i = w; i < n; i += t) body(i);
    });
  for (auto& th : pool) th.join();
}

double default_scale(int d) { return 1.0 / std::sqrt((double)d); }

// [Wiki] §一.2 / the softmax definition: one query row q[D] over m keys, key j
// at k + j * stride (its value at v + j * stride).  visible[j] == 0 excludes
// key j.  s_j = scale * q.k_j; mx = max of the visible s_j; w_j = exp(s_j - mx);
// out = sum_j w_j v_j / sum_j w_j.
void attend_row(const double* q, const double* k, const double* v, int64_t stride, int m,
                const unsigned char* visible, int d, double scale, double* out) {
  std::vector<double> s(m, 0.0);
  double mx = -std::numeric_limits<double>::infinity();
  for (int j = 0; j < m; ++j) {
    if (!visible[j]) continue;
    double dot = 0.0;
    for (int t = 0; t < d; ++t) dot += q[t] * k[j * stride + t];
    s[j] = scale * dot;
    mx = std::max(mx, s[j]);
  }
  double z = 0.0;
  for (int t = 0; t < d; ++t) out[t] = 0.0;
  for (int j = 0; j < m; ++j) {
    if (!visible[j]) continue;
    const double w = std::exp(s[j] - mx);
    z += w;
    for (int t = 0; t < d; ++t) out[t] += w * v[j * stride + t];
  }
  for (int t = 0; t < d; ++t) out[t] /= z;
}

// [Horizon] §4: the mask is added to the scores of every slot; nothing is excluded.
void attend_row_additive(const double* q, const double* k, const double* v, int64_t stride, int m,
                         const double* mask, int d, double scale, double* out) {
  std::vector<double> s(m);
  double mx = -std::numeric_limits<double>::infinity();
  for (int j = 0; j < m; ++j) {
    double dot = 0.0;
    for (int t = 0; t < d; ++t) dot += q[t] * k[j * stride + t];
    s[j] = scale * dot + mask[j];
    mx = std::max(mx, s[j]);
  }
  double z = 0.0;
  for (int t = 0; t < d; ++t) out[t] = 0.0;
  for (int j = 0; j < m; ++j) {
    const double w = std::exp(s[j] - mx);
    z += w;
    for (int t = 0; t < d; ++t) out[t] += w * v[j * stride + t];
  }
  for (int t = 0; t < d; ++t) out[t] /= z;
}

// [Wiki] §一.2: rows [0, r) of a chunk at absolute positions past + i; row i,
// query head h sees keys [0, past + i] of KV head h / (hq / hkv).  Keys of KV
// head g: key j at kv + j * key_stride + g * head_stride.
void chunk_rows(const double* q, int r, int hq, int hkv, int d, const double* k, const double* v,
                int64_t key_stride, int64_t head_stride, int past, double scale, double* out) {
  const int group = hq / hkv;
  for_each_index((int64_t)r * hq, [&](int64_t idx) {
    const int i = (int)(idx / hq), h = (int)(idx % hq);
    const int g = h / group;
    const int m = past + i + 1;
    std::vector<unsigned char> vis(m, 1);
    attend_row(q + ((int64_t)i * hq + h) * d, k + g * head_stride, v + g * head_stride, key_stride, m, vis.data(),
               d, scale, out + ((int64_t)i * hq + h) * d);
  });
}

// [Wiki] §一.1: row t of sequence b goes to slot past[b] + t of every KV head.
// cache [B, hkv, cap, d]; rows [B, r, hkv, d].  Returns -1 past the capacity.
int append_rows(double* cache, const double* rows, int b_n, int r, int hkv, int cap, int d, const int* past) {
  for (int b = 0; b < b_n; ++b) {
    if (past[b] < 0 || past[b] + r > cap) return -1;
    for (int t = 0; t < r; ++t)
      for (int g = 0; g < hkv; ++g)
        std::memcpy(cache + (((int64_t)b * hkv + g) * cap + past[b] + t) * d,
                    rows + (((int64_t)b * r + t) * hkv + g) * d, sizeof(double) * d);
  }
  return 0;
}

}  // namespace

extern "C" {

void cpo_set_threads(int n) { g_threads = n; }
int cpo_threads() { return thread_count(); }

// ---------------------------------------------------------------- integer plans

// [Wiki] §二/§三: chunks of W, the last takes the remainder.  Writes up to `cap`
// sizes; returns the count, or -1 on invalid arguments.
int cpo_chunk_plan(int n, int w, int* sizes, int cap) {
  if (w <= 0 || n < 0) return -1;
  int count = 0;
  for (int start = 0; start < n; start += w) {
    if (count < cap) sizes[count] = std::min(w, n - start);
    ++count;
  }
  return count;
}

// [Wiki] §四/§六: tiers step, 2*step, 3*step capped at W, step = ceil(W / 3),
// duplicates listed once.  Returns the number of tiers (1..3) or -1.
int cpo_query_ladder(int w, int* tiers) {
  if (w <= 0) return -1;
  const int step = (w + 2) / 3;
  int n = 0;
  for (int i = 1; i <= 3; ++i) {
    const int t = std::min(i * step, w);
    bool seen = false;
    for (int j = 0; j < n; ++j) seen = seen || tiers[j] == t;
    if (!seen) tiers[n++] = t;
  }
  return n;
}

// [Wiki] §四: the smallest tier that holds r rows; -1 unless 1 <= r <= W.
int cpo_query_width(int r, int w) {
  if (w <= 0 || r < 1 || r > w) return -1;
  int tiers[3];
  const int n = cpo_query_ladder(w, tiers);
  for (int j = 0; j < n; ++j)
    if (tiers[j] >= r) return tiers[j];
  return -1;
}

// [Horizon] §5: the aligned length, n_real rounded up to a multiple of c.
int cpo_left_pad_length(int n_real, int c) { return c > 0 ? (n_real + c - 1) / c * c : -1; }

// [Glossary] "How chunked prefill works": each step gives one row to every
// running decode, then fills the rest of the budget with chunks of waiting
// prompts in arrival order; a prompt continues next step where it stopped; a
// prompt whose last token was scheduled decodes from the next step.  Entries
// (step, seq, start, rows): start = -1 marks a decode row; decodes come first
// in each step, in sequence order.  Writes up to `cap` entries; returns the
// count, -1 on invalid arguments, -2 when the budget leaves no prompt room.
int cpo_schedule(int budget, int n_running, const int* prompt_lens, int n_prompts, int* entries, int cap) {
  if (budget <= 0 || n_running < 0 || n_prompts < 0) return -1;
  std::vector<int> decodes;
  for (int s = 0; s < n_running; ++s) decodes.push_back(s);
  std::vector<int> done(n_prompts, 0);
  int count = 0;
  auto emit = [&](int step, int seq, int start, int rows) {
    if (count < cap) {
      entries[4 * count + 0] = step;
      entries[4 * count + 1] = seq;
      entries[4 * count + 2] = start;
      entries[4 * count + 3] = rows;
    }
    ++count;
  };
  for (int step = 0;; ++step) {
    bool waiting = false;
    for (int i = 0; i < n_prompts; ++i) waiting = waiting || done[i] < prompt_lens[i];
    if (!waiting) break;
    int left = budget - (int)decodes.size();
    if (left <= 0) return -2;
    for (int s : decodes) emit(step, s, -1, 1);
    std::vector<int> finished;
    for (int i = 0; i < n_prompts && left > 0; ++i) {
      if (done[i] >= prompt_lens[i]) continue;
      const int take = std::min(left, prompt_lens[i] - done[i]);
      emit(step, n_running + i, done[i], take);
      done[i] += take;
      left -= take;
      if (done[i] == prompt_lens[i]) finished.push_back(n_running + i);
    }
    for (int s : finished) decodes.push_back(s);
  }
  return count;
}

// [Wiki] §四: x [r, e] widened to [rp, e] by repeating row r - 1.
int cpo_pad_rows(const double* x, int r, int64_t e, int rp, double* out) {
  if (r < 1 || rp < r) return -1;
  std::memcpy(out, x, sizeof(double) * r * e);
  for (int t = r; t < rp; ++t) std::memcpy(out + t * e, x + (int64_t)(r - 1) * e, sizeof(double) * e);
  return 0;
}

// ---------------------------------------------------------------- attention

// One chunk over a cache in position order: q [r, hq, d] at positions
// past .. past + r - 1; k_seq / v_seq [n, hkv, d] with n >= past + r.
// scale <= 0 means 1/sqrt(d).  out [r, hq, d].
void cpo_chunk_attention(const double* q, int r, int hq, int hkv, int d, const double* k_seq, const double* v_seq,
                         int past, double scale, double* out) {
  if (scale <= 0) scale = default_scale(d);
  chunk_rows(q, r, hq, hkv, d, k_seq, v_seq, (int64_t)hkv * d, d, past, scale, out);
}

// [Glossary] example, the one-shot branch: causal attention of n rows.
void cpo_causal_attention(const double* q, int n, int hq, int hkv, int d, const double* k, const double* v,
                          double scale, double* out) {
  cpo_chunk_attention(q, n, hq, hkv, d, k, v, 0, scale, out);
}

// [Wiki] §一.1, [Glossary] example, the chunk loop: a cache [hkv, cap, d]
// starts zero; for each chunk of chunk_plan(n, W) its K/V rows are appended at
// slots [start, start + r) and its rows attend to the cache.  out [n, hq, d];
// k_cache / v_cache [hkv, cap, d] receive the final cache; snaps (may be null)
// receive [nchunks, 2, hkv, cap, d] (K then V after each chunk).  Returns the
// number of chunks, or -1 on invalid arguments.
int cpo_chunked_prefill(const double* q, const double* k, const double* v, int n, int hq, int hkv, int d, int w,
                        int cap, double scale, double* out, double* k_cache, double* v_cache, double* snaps) {
  if (w <= 0 || cap < n || hq % hkv) return -1;
  if (scale <= 0) scale = default_scale(d);
  const int64_t cache_elems = (int64_t)hkv * cap * d;
  std::fill(k_cache, k_cache + cache_elems, 0.0);
  std::fill(v_cache, v_cache + cache_elems, 0.0);
  std::vector<int> sizes((size_t)std::max(1, (n + w - 1) / w));
  const int nchunks = cpo_chunk_plan(n, w, sizes.data(), (int)sizes.size());
  int start = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int r = sizes[c];
    append_rows(k_cache, k + (int64_t)start * hkv * d, 1, r, hkv, cap, d, &start);
    append_rows(v_cache, v + (int64_t)start * hkv * d, 1, r, hkv, cap, d, &start);
    // Cache layout [hkv, cap, d]: key j of head g at (g * cap + j) * d.
    chunk_rows(q + (int64_t)start * hq * d, r, hq, hkv, d, k_cache, v_cache, d, (int64_t)cap * d, start, scale,
               out + (int64_t)start * hq * d);
    if (snaps) {
      std::memcpy(snaps + (2 * (int64_t)c) * cache_elems, k_cache, sizeof(double) * cache_elems);
      std::memcpy(snaps + (2 * (int64_t)c + 1) * cache_elems, v_cache, sizeof(double) * cache_elems);
    }
    start += r;
  }
  return nchunks;
}

// [Wiki] §一.1: contiguous append in place.  cache [b, hkv, cap, d]; rows
// [b, r, hkv, d]; past [b].  Returns -1 when a row would pass the capacity.
int cpo_kv_append(double* cache, const double* rows, int b, int r, int hkv, int cap, int d, const int* past) {
  return append_rows(cache, rows, b, r, hkv, cap, d, past);
}

// [Wiki] §四: one padded chunk.  The r real rows widen to rp = query_width(r, W)
// rows (copies of the last real row); all rp rows are appended at past and
// attend; the caller keeps out rows [0, r) and rewinds the length to past + r.
// kc / vc [hkv, cap, d] in place; q_pad [rp, hq, d] of scratch; out [rp, hq, d].
// Returns rp, or -1 on invalid arguments.
int cpo_padded_chunk(const double* q_real, const double* k_real, const double* v_real, int r, int hq, int hkv,
                     int d, double* kc, double* vc, int cap, int past, int w, double scale, double* out) {
  const int rp = cpo_query_width(r, w);
  if (rp < 0 || past + rp > cap) return -1;
  if (scale <= 0) scale = default_scale(d);
  std::vector<double> qp((size_t)rp * hq * d), kp((size_t)rp * hkv * d), vp((size_t)rp * hkv * d);
  cpo_pad_rows(q_real, r, (int64_t)hq * d, rp, qp.data());
  cpo_pad_rows(k_real, r, (int64_t)hkv * d, rp, kp.data());
  cpo_pad_rows(v_real, r, (int64_t)hkv * d, rp, vp.data());
  append_rows(kc, kp.data(), 1, rp, hkv, cap, d, &past);
  append_rows(vc, vp.data(), 1, rp, hkv, cap, d, &past);
  chunk_rows(qp.data(), rp, hq, hkv, d, kc, vc, d, (int64_t)cap * d, past, scale, out);
  return rp;
}

// ---------------------------------------------------------------- rolling cache

// [Horizon] §3: cat(cache, new) along the sequence, minus the oldest c rows.
// cache [h, C, d] and new [h, c, d]; out [h, C, d] (may not alias cache).
void cpo_rolling_update(const double* cache, const double* fresh, int h, int cap, int c, int d, double* out) {
  for (int hh = 0; hh < h; ++hh)
    for (int j = 0; j < cap; ++j) {
      // slot j of the concatenation [cache ; new] after dropping its first c rows
      const int src = j + c;
      const double* row = src < cap ? cache + ((int64_t)hh * cap + src) * d
                                    : fresh + ((int64_t)hh * c + (src - cap)) * d;
      std::memcpy(out + ((int64_t)hh * cap + j) * d, row, sizeof(double) * d);
    }
}

// [Horizon] §4: mask [c, C] for chunk k: row i is position p = k*c + i; slot j
// holds position a = (k+1)*c - C + j; 0 where a >= 0, a >= left_pad and a <= p,
// else -32768.
void cpo_rolling_mask(int c, int cap, int k, int left_pad, double* out) {
  for (int i = 0; i < c; ++i) {
    const int p = k * c + i;
    for (int j = 0; j < cap; ++j) {
      const int a = (k + 1) * c - cap + j;
      out[(int64_t)i * cap + j] = (a >= 0 && a >= left_pad && a <= p) ? 0.0 : -32768.0;
    }
  }
}

// [Horizon] §3-§5: rolling prefill of the left-padded sequence q/k/v [L, h, d]
// (L a multiple of c, c <= C).  Per chunk: roll its K/V into the [h, C, d]
// cache (zero at the start), build the mask, attend over all C slots with the
// mask added.  out [L, h, d]; snaps (may be null) [L/c, 2, h, C, d].
// Returns the number of chunks or -1.
int cpo_rolling_prefill(const double* q, const double* k, const double* v, int L, int h, int d, int c, int cap,
                        int left_pad, double scale, double* out, double* snaps) {
  if (c <= 0 || L % c || c > cap) return -1;
  if (scale <= 0) scale = default_scale(d);
  const int64_t elems = (int64_t)h * cap * d;
  std::vector<double> kc(elems, 0.0), vc(elems, 0.0), tmp(elems), fresh((size_t)h * c * d);
  std::vector<double> mask((size_t)c * cap);
  for (int ci = 0; ci < L / c; ++ci) {
    for (int pass = 0; pass < 2; ++pass) {
      const double* src = pass == 0 ? k : v;
      std::vector<double>& cache = pass == 0 ? kc : vc;
      for (int hh = 0; hh < h; ++hh)  // the chunk's rows as [h, c, d]
        for (int t = 0; t < c; ++t)
          std::memcpy(fresh.data() + ((int64_t)hh * c + t) * d, src + ((int64_t)(ci * c + t) * h + hh) * d,
                      sizeof(double) * d);
      cpo_rolling_update(cache.data(), fresh.data(), h, cap, c, d, tmp.data());
      cache.swap(tmp);
    }
    cpo_rolling_mask(c, cap, ci, left_pad, mask.data());
    for_each_index((int64_t)c * h, [&](int64_t idx) {
      const int i = (int)(idx / h), hh = (int)(idx % h);
      const int p = ci * c + i;
      attend_row_additive(q + ((int64_t)p * h + hh) * d, kc.data() + (int64_t)hh * cap * d,
                          vc.data() + (int64_t)hh * cap * d, d, cap, mask.data() + (int64_t)i * cap, d, scale,
                          out + ((int64_t)p * h + hh) * d);
    });
    if (snaps) {
      std::memcpy(snaps + (2 * (int64_t)ci) * elems, kc.data(), sizeof(double) * elems);
      std::memcpy(snaps + (2 * (int64_t)ci + 1) * elems, vc.data(), sizeof(double) * elems);
    }
  }
  return L / c;
}

// ---------------------------------------------------------------- paged cache

// [Glossary] "Related techniques" (PagedAttention): the token at absolute
// position pos of a sequence lives in page table_row[pos / page] at offset
// pos % page.  pool [num_pages, hkv, page, d]; row [hkv, d].
int cpo_paged_write(double* pool, int num_pages, int hkv, int page, int d, const int* table_row, int pos,
                    const double* row) {
  const int pg = table_row[pos / page];
  if (pg < 0 || pg >= num_pages) return -1;
  for (int g = 0; g < hkv; ++g)
    std::memcpy(pool + (((int64_t)pg * hkv + g) * page + pos % page) * d, row + (int64_t)g * d, sizeof(double) * d);
  return 0;
}

// The first n positions of a paged sequence in position order: out [n, hkv, d].
int cpo_paged_gather(const double* pool, int num_pages, int hkv, int page, int d, const int* table_row, int n,
                     double* out) {
  for (int a = 0; a < n; ++a) {
    const int pg = table_row[a / page];
    if (pg < 0 || pg >= num_pages) return -1;
    for (int g = 0; g < hkv; ++g)
      std::memcpy(out + ((int64_t)a * hkv + g) * d, pool + (((int64_t)pg * hkv + g) * page + a % page) * d,
                  sizeof(double) * d);
  }
  return 0;
}

// [Glossary] "How chunked prefill works": one token-budget step.  Sequence s
// owns rows[s] consecutive rows of q [T, hq, d] and k_new / v_new [T, hkv, d].
// Every row's K/V is written at positions past[s] .. past[s] + rows[s] - 1 of
// its pages first (pools updated in place); then each sequence's rows attend
// as one chunk over its gathered cache.  table [S, max_blocks].  out [T, hq, d];
// past is advanced by rows.  Returns 0, or -1 on a page id out of range.
int cpo_mixed_step(const double* q, const double* k_new, const double* v_new, double* k_pool, double* v_pool,
                   int num_pages, int hq, int hkv, int page, int d, const int* table, int max_blocks, const int* rows,
                   int* past, int num_seqs, double scale, double* out) {
  if (scale <= 0) scale = default_scale(d);
  int64_t t = 0;
  for (int s = 0; s < num_seqs; ++s) {
    for (int i = 0; i < rows[s]; ++i) {
      if (cpo_paged_write(k_pool, num_pages, hkv, page, d, table + (int64_t)s * max_blocks, past[s] + i,
                          k_new + (t + i) * hkv * d) ||
          cpo_paged_write(v_pool, num_pages, hkv, page, d, table + (int64_t)s * max_blocks, past[s] + i,
                          v_new + (t + i) * hkv * d))
        return -1;
    }
    t += rows[s];
  }
  t = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int n = past[s] + rows[s];
    std::vector<double> ks((size_t)n * hkv * d), vs((size_t)n * hkv * d);
    if (cpo_paged_gather(k_pool, num_pages, hkv, page, d, table + (int64_t)s * max_blocks, n, ks.data()) ||
        cpo_paged_gather(v_pool, num_pages, hkv, page, d, table + (int64_t)s * max_blocks, n, vs.data()))
      return -1;
    cpo_chunk_attention(q + t * hq * d, rows[s], hq, hkv, d, ks.data(), vs.data(), past[s], scale,
                        out + t * hq * d);
    t += rows[s];
  }
  for (int s = 0; s < num_seqs; ++s) past[s] += rows[s];
  return 0;
}

}  // extern "C"
