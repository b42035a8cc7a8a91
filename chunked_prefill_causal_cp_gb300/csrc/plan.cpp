// plan.cpp -- host-side integer helpers of the C ABI: chunk plan, query-width
// ladder, aligned length, rolling mask, token-budget scheduler, status text.
// Integer-exact; no GPU work.
#include <cstdint>
#include <vector>

#include "../../include/cp_api.h"

extern "C" {

// [Wiki] 三: chunks of width `chunk`, the last one takes the remainder.
int32_t cp_chunk_plan(int32_t n_tokens, int32_t chunk, int32_t* sizes, int32_t cap) {
  if (n_tokens < 0 || chunk <= 0 || cap < 0 || (cap > 0 && sizes == nullptr)) return CP_ERR_INVALID_ARG;
  int32_t count = 0;
  for (int64_t start = 0; start < n_tokens; start += chunk) {
    const int64_t left = (int64_t)n_tokens - start;
    if (count < cap) sizes[count] = (int32_t)(left < chunk ? left : chunk);
    ++count;
  }
  return count;
}

// [Wiki] 四 / 六: tiers step, 2*step, 3*step with step = ceil(chunk/3), capped
// at chunk so the top tier is exactly the chunk width; duplicates dropped.
int32_t cp_query_ladder(int32_t chunk, int32_t* tiers) {
  if (chunk <= 0 || tiers == nullptr) return CP_ERR_INVALID_ARG;
  const int32_t step = (chunk + 2) / 3;
  int32_t count = 0;
  for (int32_t i = 1; i <= 3; ++i) {
    int64_t t = (int64_t)i * step;
    if (t > chunk) t = chunk;
    if (count == 0 || tiers[count - 1] != (int32_t)t) tiers[count++] = (int32_t)t;
  }
  return count;
}

int32_t cp_query_width(int32_t real_rows, int32_t chunk) {
  if (chunk <= 0 || real_rows < 1 || real_rows > chunk) return CP_ERR_INVALID_ARG;
  int32_t tiers[3];
  const int32_t n = cp_query_ladder(chunk, tiers);
  for (int32_t i = 0; i < n; ++i)
    if (tiers[i] >= real_rows) return tiers[i];
  return CP_ERR_INVALID_ARG;
}

// [Horizon] 5: left-pad to a multiple of the chunk size.
int32_t cp_aligned_length(int32_t n_real, int32_t c) {
  if (n_real < 0 || c <= 0) return CP_ERR_INVALID_ARG;
  const int64_t L = ((int64_t)n_real + c - 1) / c * c;
  return L > INT32_MAX ? CP_ERR_INVALID_ARG : (int32_t)L;
}

// [Horizon] 4: rows cut from the causal mask, key axis right-aligned to C,
// left-filled with -32768; pad positions and unwritten slots masked too.
int cp_rolling_mask(int32_t c, int32_t C, int32_t chunk_idx, int32_t left_pad, float* out) {
  if (c <= 0 || C <= 0 || c > C || chunk_idx < 0 || left_pad < 0 || out == nullptr) return CP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < c; ++i) {
    const int64_t p = (int64_t)chunk_idx * c + i;
    for (int32_t j = 0; j < C; ++j) {
      const int64_t a = ((int64_t)chunk_idx + 1) * c - C + j;
      const bool ok = a >= 0 && a >= left_pad && a <= p;
      out[(int64_t)i * C + j] = ok ? 0.0f : -32768.0f;
    }
  }
  return CP_OK;
}

// [Glossary] "How chunked prefill works": decodes first, then waiting prompt
// chunks in arrival order until the budget is spent; a prompt decodes from
// the step after its last chunk.
int32_t cp_schedule(int32_t budget, int32_t n_running, const int32_t* prompt_lens, int32_t n_prompts,
                    cp_sched_entry* out, int32_t cap) {
  if (budget <= 0 || n_running < 0 || n_prompts < 0 || cap < 0 || (n_prompts > 0 && prompt_lens == nullptr) ||
      (cap > 0 && out == nullptr))
    return CP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_prompts; ++i)
    if (prompt_lens[i] < 0) return CP_ERR_INVALID_ARG;
  std::vector<int32_t> done(n_prompts, 0);
  std::vector<int32_t> decodes;
  for (int32_t i = 0; i < n_running; ++i) decodes.push_back(i);
  int32_t count = 0;
  auto emit = [&](int32_t step, int32_t seq, int32_t start, int32_t rows) {
    if (count < cap) out[count] = cp_sched_entry{step, seq, start, rows};
    ++count;
  };
  for (int32_t step = 0;; ++step) {
    bool pending = false;
    for (int32_t i = 0; i < n_prompts; ++i) pending |= done[i] < prompt_lens[i];
    if (!pending) break;
    int64_t left = (int64_t)budget - (int64_t)decodes.size();
    if (left <= 0) return CP_ERR_INVALID_ARG;
    for (int32_t sid : decodes) emit(step, sid, -1, 1);
    std::vector<int32_t> finished;
    for (int32_t i = 0; i < n_prompts && left > 0; ++i) {
      if (done[i] >= prompt_lens[i]) continue;
      const int32_t rest = prompt_lens[i] - done[i];
      const int32_t take = (int32_t)(left < rest ? left : rest);
      emit(step, n_running + i, done[i], take);
      done[i] += take;
      left -= take;
      if (done[i] == prompt_lens[i]) finished.push_back(n_running + i);
    }
    for (int32_t sid : finished) decodes.push_back(sid);
  }
  return count;
}

const char* cp_status_string(int32_t status) {
  switch (status) {
    case CP_OK: return "ok";
    case CP_ERR_INVALID_ARG: return "invalid argument";
    case CP_ERR_UNSUPPORTED: return "unsupported configuration";
    case CP_ERR_CAPACITY: return "rows do not fit in the cache";
    case CP_ERR_CUDA: return "CUDA error";
    case CP_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int32_t cp_abi_version(void) { return CP_ABI_VERSION; }

}  // extern "C"
