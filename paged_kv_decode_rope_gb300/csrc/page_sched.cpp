// page_sched.cpp -- host page allocator and page-budget admission (pkv_sched.h).
//
// The policy is the one "Hours of YouTube and 85 handtyped pages of notes on
// LLM Inference – Start here" describes for its continuous batching: budgets
// are reserved at admission and pages are handed out lazily; see pkv_sched.h.
// Plain host C++17, deterministic for a given seed on any platform: the free
// list is shuffled with a Fisher-Yates pass driven by splitmix64.
#include <cerrno>
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "../../include/pkv_sched.h"

namespace {

constexpr int kPageTokens = 16;

struct Request {
  int prompt = 0;
  int max_new = 0;       // after clamping to the context
  int budget_tokens = 0; // largest processed prefix: prompt + max_new - 1
  int credits = 0;       // pages over all layers reserved at admission
  bool active = false;
  bool finished = false;
  bool waited = false;
  std::vector<std::vector<int32_t>> pages;  // [layer] -> page ids in token order
};

uint64_t splitmix64(uint64_t& x) {
  uint64_t z = (x += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int pages_for(int tokens) { return (tokens + kPageTokens - 1) / kPageTokens; }

}  // namespace

struct pkv_sched {
  int num_pages = 0;
  int num_layers = 0;
  int context = 0;
  bool static_mode = false;
  std::vector<int32_t> free_list;  // a stack: the next page handed out is the back
  std::vector<Request> reqs;       // indexed by request id
  std::deque<int> queue;           // waiting request ids, FIFO
  int reserved = 0;
  int assigned = 0;
  int active = 0;
  pkv_sched_stats_t st = {};
};

namespace {

int credits_for(const pkv_sched* s, int prompt, int max_new, int* clamped_new, int* budget_tokens) {
  int m = max_new;
  if (prompt + m > s->context) m = s->context - prompt;
  const int tokens = prompt + m - 1;
  if (clamped_new) *clamped_new = m;
  if (budget_tokens) *budget_tokens = tokens;
  return pages_for(tokens) * s->num_layers;
}

bool valid_active(const pkv_sched* s, int id) {
  return id >= 0 && id < static_cast<int>(s->reqs.size()) && s->reqs[id].active;
}

}  // namespace

extern "C" {

int pkv_sched_create(pkv_sched_t** out, int num_pages, int num_layers, int context_len,
                     int static_batching, uint64_t seed) {
  if (!out || num_pages < 1 || num_layers < 1 || context_len < 2) return -EINVAL;
  pkv_sched* s = new (std::nothrow) pkv_sched;
  if (!s) return -ENOMEM;
  s->num_pages = num_pages;
  s->num_layers = num_layers;
  s->context = context_len;
  s->static_mode = static_batching != 0;
  s->free_list.resize(num_pages);
  // The stack hands out its back first: store ids descending so that an
  // unshuffled list gives pages 0, 1, 2, ...
  for (int i = 0; i < num_pages; ++i) s->free_list[i] = num_pages - 1 - i;
  if (seed != 0) {
    uint64_t x = seed;
    for (int i = num_pages - 1; i > 0; --i) {
      const int j = static_cast<int>(splitmix64(x) % static_cast<uint64_t>(i + 1));
      const int32_t t = s->free_list[i];
      s->free_list[i] = s->free_list[j];
      s->free_list[j] = t;
    }
  }
  s->st.pool_pages = num_pages;
  *out = s;
  return 0;
}

int pkv_sched_destroy(pkv_sched_t* s) {
  if (!s) return -EINVAL;
  delete s;
  return 0;
}

int pkv_sched_budget(const pkv_sched_t* s, int prompt_len, int max_new) {
  if (!s || prompt_len < 1 || prompt_len >= s->context || max_new < 1) return -EINVAL;
  return credits_for(s, prompt_len, max_new, nullptr, nullptr);
}

int pkv_sched_submit(pkv_sched_t* s, int prompt_len, int max_new, int* request_id) {
  if (!s || !request_id || prompt_len < 1 || prompt_len >= s->context || max_new < 1) return -EINVAL;
  Request r;
  r.prompt = prompt_len;
  r.credits = credits_for(s, prompt_len, max_new, &r.max_new, &r.budget_tokens);
  if (r.credits > s->num_pages) {
    ++s->st.rejected;
    return -ENOSPC;
  }
  r.pages.resize(s->num_layers);
  const int id = static_cast<int>(s->reqs.size());
  s->reqs.push_back(std::move(r));
  s->queue.push_back(id);
  *request_id = id;
  return 0;
}

int pkv_sched_admit(pkv_sched_t* s, int* ids, int max_ids) {
  if (!s || max_ids < 0 || (max_ids > 0 && !ids)) return -EINVAL;
  int n = 0;
  if (!s->static_mode || s->active == 0) {
    while (!s->queue.empty() && n < max_ids) {
      Request& r = s->reqs[s->queue.front()];
      if (r.credits > s->num_pages - s->reserved) break;  // FIFO: the head waits, so do all behind it
      r.active = true;
      s->reserved += r.credits;
      ++s->active;
      ++s->st.admitted;
      ids[n++] = s->queue.front();
      s->queue.pop_front();
    }
    if (s->active > s->st.peak_active) s->st.peak_active = s->active;
  }
  for (int id : s->queue) {
    Request& r = s->reqs[id];
    if (!r.waited) {
      r.waited = true;
      ++s->st.admission_waits;
    }
  }
  return n;
}

int pkv_sched_grow(pkv_sched_t* s, int request_id, int kv_len) {
  if (!s || !valid_active(s, request_id) || kv_len < 0) return -EINVAL;
  Request& r = s->reqs[request_id];
  if (kv_len > r.budget_tokens) return -EINVAL;
  const int need = pages_for(kv_len);
  for (auto& row : r.pages) {
    while (static_cast<int>(row.size()) < need) {
      // Credits cover every page a request can reach, so the list cannot be empty here.
      if (s->free_list.empty()) return -ENOSPC;
      row.push_back(s->free_list.back());
      s->free_list.pop_back();
      ++s->assigned;
    }
  }
  if (s->assigned > s->st.peak_assigned_pages) s->st.peak_assigned_pages = s->assigned;
  return 0;
}

int pkv_sched_block_row(const pkv_sched_t* s, int request_id, int layer, int32_t* row,
                        int max_blocks) {
  if (!s || !valid_active(s, request_id) || layer < 0 || layer >= s->num_layers || !row ||
      max_blocks < 0)
    return -EINVAL;
  const auto& pages = s->reqs[request_id].pages[layer];
  const int n = static_cast<int>(pages.size());
  if (n > max_blocks) return -EINVAL;
  for (int i = 0; i < max_blocks; ++i) row[i] = i < n ? pages[i] : -1;
  return n;
}

int pkv_sched_finish(pkv_sched_t* s, int request_id) {
  if (!s || !valid_active(s, request_id)) return -EINVAL;
  Request& r = s->reqs[request_id];
  for (auto& row : r.pages) {
    for (int32_t p : row) s->free_list.push_back(p);
    s->assigned -= static_cast<int>(row.size());
    row.clear();
  }
  s->reserved -= r.credits;
  r.active = false;
  r.finished = true;
  --s->active;
  ++s->st.completed;
  return 0;
}

int pkv_sched_note_batch(pkv_sched_t* s, int batch) {
  if (!s || batch < 0) return -EINVAL;
  if (batch > s->st.largest_batch) s->st.largest_batch = batch;
  return 0;
}

int pkv_sched_stats(const pkv_sched_t* s, pkv_sched_stats_t* out) {
  if (!s || !out) return -EINVAL;
  *out = s->st;
  out->free_pages = static_cast<int>(s->free_list.size());
  out->assigned_pages = s->assigned;
  out->reserved_credits = s->reserved;
  out->active = s->active;
  out->waiting = static_cast<int>(s->queue.size());
  return 0;
}

}  // extern "C"
