// KV-cache allocator simulator: a contiguous allocator and a paged allocator
// serving the same request stream ("10 — Paged Attention" tutorial, §10
// exercises B and C: fragmentation, allocation failures, concurrency, block-size
// sweep).  The step rules are spelled out in the header; every quantity is an
// integer sum over steps.
#include <stdint.h>

#include <deque>
#include <iterator>
#include <map>
#include <vector>

#include "../../include/pagedattn.h"

namespace {

int64_t next_pow2(int64_t x) {
  int64_t p = 1;
  while (p < x) p *= 2;
  return p;
}

// Free extents of a linear space by start address; first fit, merge on free.
class FirstFit {
 public:
  explicit FirstFit(int64_t capacity) {
    if (capacity > 0) free_[0] = capacity;
    total_ = capacity > 0 ? capacity : 0;
  }
  int64_t total_free() const { return total_; }
  bool allocate(int64_t size, int64_t* start) {
    for (auto it = free_.begin(); it != free_.end(); ++it) {
      if (it->second >= size) {
        *start = it->first;
        const int64_t rest = it->second - size, at = it->first + size;
        free_.erase(it);
        if (rest > 0) free_[at] = rest;
        total_ -= size;
        return true;
      }
    }
    return false;
  }
  void release(int64_t start, int64_t size) {
    auto it = free_.emplace(start, size).first;
    total_ += size;
    auto next = std::next(it);
    if (next != free_.end() && it->first + it->second == next->first) {
      it->second += next->second;
      free_.erase(next);
    }
    if (it != free_.begin()) {
      auto prev = std::prev(it);
      if (prev->first + prev->second == it->first) {
        prev->second += it->second;
        free_.erase(it);
      }
    }
  }

 private:
  std::map<int64_t, int64_t> free_;
  int64_t total_ = 0;
};

}  // namespace

extern "C" pa_status pa_sim_run(const pa_sim_config* cfg, const int32_t* arrival_step,
                                const int32_t* prompt_len, const int32_t* output_len,
                                int num_requests, pa_sim_result* out) {
  if (!cfg || !out || num_requests < 0 ||
      (num_requests > 0 && (!arrival_step || !prompt_len || !output_len)))
    return PA_ERR_INVALID_ARG;
  const bool paged = cfg->allocator == PA_SIM_PAGED;
  if (!paged && cfg->allocator != PA_SIM_CONTIGUOUS) return PA_ERR_INVALID_ARG;
  if (cfg->reserve < PA_SIM_RESERVE_MAX || cfg->reserve > PA_SIM_RESERVE_EXACT)
    return PA_ERR_INVALID_ARG;
  if (cfg->capacity_tokens < 0 || cfg->max_seq_len < 2 || cfg->max_steps < 0 ||
      (paged && cfg->block_size <= 0))
    return PA_ERR_INVALID_ARG;
  const int n = num_requests;
  const int64_t bs = paged ? cfg->block_size : 1;
  auto reservation = [&](int r) -> int64_t {
    const int64_t total = (int64_t)prompt_len[r] + output_len[r];
    if (cfg->reserve == PA_SIM_RESERVE_MAX) return cfg->max_seq_len;
    if (cfg->reserve == PA_SIM_RESERVE_POW2) return next_pow2(total);
    return total;
  };
  for (int i = 0; i < n; ++i) {
    if (prompt_len[i] < 1 || output_len[i] < 1 ||
        (int64_t)prompt_len[i] + output_len[i] > cfg->max_seq_len)
      return PA_ERR_INVALID_ARG;
    if (i > 0 && arrival_step[i] < arrival_step[i - 1]) return PA_ERR_INVALID_ARG;
    const int64_t total = (int64_t)prompt_len[i] + output_len[i];
    if (paged ? (total + bs - 1) / bs > cfg->capacity_tokens / bs
              : reservation(i) > cfg->capacity_tokens)
      return PA_ERR_INVALID_ARG;
  }

  std::vector<int64_t> cur(prompt_len, prompt_len + n);
  std::vector<int64_t> admitted((size_t)n, -1), start((size_t)n, 0), held((size_t)n, 0);
  FirstFit ff(paged ? 0 : cfg->capacity_tokens);
  int64_t free_blocks = paged ? cfg->capacity_tokens / bs : 0;
  std::deque<int> waiting;
  std::vector<int> running, kept, preempted;
  pa_sim_result res = {};
  int next = 0;
  int64_t t = 0;
  while (res.completed < n && t < cfg->max_steps) {
    while (next < n && arrival_step[next] <= t) waiting.push_back(next++);
    // admission, first come first served
    while (!waiting.empty()) {
      const int r = waiting.front();
      bool ok;
      if (paged) {
        const int64_t need = (cur[r] + bs - 1) / bs;
        ok = free_blocks >= need;
        if (ok) {
          free_blocks -= need;
          held[r] = need;
        }
      } else {
        const int64_t need = reservation(r);
        int64_t at = 0;
        ok = ff.allocate(need, &at);
        if (ok) {
          start[r] = at;
          held[r] = need;
        } else if (ff.total_free() >= need) {
          ++res.fragmentation_failures;
        }
      }
      if (!ok) {
        ++res.failed_allocations;
        break;
      }
      waiting.pop_front();
      running.push_back(r);
      admitted[r] = t;
    }
    // growth: one token per request admitted in an earlier step
    kept.clear();
    preempted.clear();
    for (int r : running) {
      if (admitted[r] != t) {
        if (paged && cur[r] % bs == 0) {
          if (free_blocks == 0) {
            ++res.failed_allocations;
            ++res.preemptions;
            free_blocks += held[r];
            held[r] = 0;
            preempted.push_back(r);
            continue;
          }
          --free_blocks;
          ++held[r];
        }
        ++cur[r];
      }
      kept.push_back(r);
    }
    running.swap(kept);
    for (auto it = preempted.rbegin(); it != preempted.rend(); ++it) waiting.push_front(*it);
    // measurement
    if (!running.empty()) {
      int64_t stored = 0, mem = 0, tl_max = 0;
      for (int r : running) {
        stored += cur[r];
        mem += paged ? held[r] * bs : held[r];
        if (paged) {
          res.sum_table_len += held[r];
          if (held[r] > tl_max) tl_max = held[r];
        }
      }
      if (tl_max > res.max_table_len) res.max_table_len = tl_max;
      ++res.busy_steps;
      res.sum_stored += stored;
      res.sum_held += mem;
      if (stored > res.peak_stored) res.peak_stored = stored;
      if (mem > res.peak_held) res.peak_held = mem;
      res.sum_concurrency += (int64_t)running.size();
      if ((int64_t)running.size() > res.max_concurrency)
        res.max_concurrency = (int64_t)running.size();
    }
    // completion
    kept.clear();
    for (int r : running) {
      if (cur[r] == (int64_t)prompt_len[r] + output_len[r]) {
        if (paged) free_blocks += held[r];
        else ff.release(start[r], held[r]);
        held[r] = 0;
        ++res.completed;
      } else {
        kept.push_back(r);
      }
    }
    running.swap(kept);
    ++t;
  }
  res.steps = t;
  *out = res;
  return PA_OK;
}
