// Two-phase continuous-batching scheduler over the block pool.
//
// PhotonInfer README, "Technical details > Continuous batching scheduler":
//   phase 1 continues every RUNNING request (no interruption), phase 2
//   admits WAITING requests into the remaining capacity; a request moves
//   WAITING -> RUNNING -> FINISHED, with preemption; num_computed_tokens marks
//   the exact point a request resumes from.  "Key features > vLLM-style
//   continuous batching": requests join at token granularity, without
//   waiting for the batch to finish.
//
// Token accounting (the plainest reading): a request knows L = prompt_len +
// num_generated tokens.  A scheduled request processes tokens
// [num_computed, L) this step -- its whole known sequence right after
// admission (prefill), one token afterwards (decode) -- and its K/V slots
// cover positions up to L - 1, so it holds ceil(L / block_size) blocks.
// After the step, num_computed = L and one more token has been generated.
//
// Preemption: when the pool cannot supply the blocks that the running
// requests need to continue, the most recently admitted running request is
// preempted -- its blocks go back to the pool, num_computed drops to 0
// (recomputed on re-admission) and it returns to the FRONT of the waiting
// queue, so preempted requests resume in their original order.  Admission is
// strictly first-come first-served: the first waiting request that does not
// fit (batch slots, token budget, free blocks) ends phase 2.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "photon.h"

namespace {

struct Request {
  int64_t id = 0;
  int32_t prompt_len = 0;
  int32_t max_new = 0;
  int32_t num_generated = 0;
  int32_t num_computed = 0;
  int32_t state = PHOTON_REQ_WAITING;
  int32_t generation = 0;  // bumped whenever its blocks are given back
  std::vector<int32_t> blocks;
  int32_t known() const { return prompt_len + num_generated; }
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct photon_scheduler {
  photon_scheduler_config cfg{};
  photon_block_pool *pool = nullptr;
  std::unordered_map<int64_t, Request> reqs;
  std::deque<int64_t> waiting;   // front first
  std::vector<int64_t> running;  // admission order
  std::vector<int64_t> stepped;  // requests of the open step
  bool step_open = false;
  // what the caller's block_tables rows held after the last emitted batch:
  // the request in each row and how many of its entries were written
  std::vector<int64_t> row_id;
  std::vector<int32_t> row_gen;
  std::vector<int32_t> row_len;
  const int32_t *last_tables = nullptr;
};

extern "C" {

int photon_scheduler_create(const photon_scheduler_config *cfg, photon_block_pool *pool,
                            photon_scheduler **out) {
  if (!cfg || !pool || !out) return PHOTON_ERR_INVALID_ARG;
  if (cfg->max_running <= 0 || cfg->max_step_tokens <= 0 || cfg->max_blocks_per_seq <= 0 ||
      cfg->block_size <= 0)
    return PHOTON_ERR_INVALID_ARG;
  photon_scheduler *s = new (std::nothrow) photon_scheduler;
  if (!s) return PHOTON_ERR_INVALID_ARG;
  s->cfg = *cfg;
  s->pool = pool;
  *out = s;
  return PHOTON_OK;
}

void photon_scheduler_destroy(photon_scheduler *s) {
  if (!s) return;
  for (auto &kv : s->reqs)
    if (!kv.second.blocks.empty())
      photon_block_pool_free(s->pool, kv.second.blocks.data(),
                             static_cast<int32_t>(kv.second.blocks.size()));
  delete s;
}

int photon_scheduler_add_request(photon_scheduler *s, int64_t request_id, int32_t prompt_len,
                                 int32_t max_new_tokens) {
  if (!s || prompt_len <= 0 || max_new_tokens <= 0) return PHOTON_ERR_INVALID_ARG;
  if (s->reqs.count(request_id)) return PHOTON_ERR_INVALID_ARG;
  const int64_t longest = static_cast<int64_t>(prompt_len) + max_new_tokens;
  const int64_t blocks = ceil_div(longest, s->cfg.block_size);
  // a request that could never run would block the first-come queue forever
  if (blocks > s->cfg.max_blocks_per_seq) return PHOTON_ERR_INVALID_ARG;
  if (blocks > photon_block_pool_num_free(s->pool) +
                   [&] {
                     int64_t held = 0;
                     for (auto &kv : s->reqs) held += static_cast<int64_t>(kv.second.blocks.size());
                     return held;
                   }())
    return PHOTON_ERR_POOL_EXHAUSTED;
  // after a preemption its whole known sequence (at most prompt + max_new - 1
  // tokens) is recomputed in one step: that must fit the step's token budget
  if (longest - 1 > s->cfg.max_step_tokens) return PHOTON_ERR_INVALID_ARG;
  Request r;
  r.id = request_id;
  r.prompt_len = prompt_len;
  r.max_new = max_new_tokens;
  s->reqs.emplace(request_id, std::move(r));
  s->waiting.push_back(request_id);
  return PHOTON_OK;
}

int photon_scheduler_schedule(photon_scheduler *s, photon_step_batch *b) {
  if (!s || !b) return PHOTON_ERR_INVALID_ARG;
  if (s->step_open) return PHOTON_ERR_INVALID_ARG;  // complete the previous step first
  if (b->max_seqs < s->cfg.max_running || b->max_tokens < s->cfg.max_step_tokens ||
      !b->request_ids || !b->num_new_tokens || !b->context_lens || !b->block_tables ||
      !b->token_seq || !b->positions || !b->slot_mapping)
    return PHOTON_ERR_INVALID_ARG;
  const int32_t bs = s->cfg.block_size;
  b->num_preempted = 0;
  b->num_admitted = 0;

  // ---- phase 1: every running request continues; preempt newest-first while
  // the pool cannot cover their next blocks
  auto extra_blocks = [&]() {
    int64_t extra = 0;
    for (int64_t id : s->running) {
      const Request &r = s->reqs[id];
      extra += std::max<int64_t>(0, ceil_div(r.known(), bs) - static_cast<int64_t>(r.blocks.size()));
    }
    return extra;
  };
  while (!s->running.empty() && extra_blocks() > photon_block_pool_num_free(s->pool)) {
    const int64_t id = s->running.back();
    s->running.pop_back();
    Request &r = s->reqs[id];
    photon_block_pool_free(s->pool, r.blocks.data(), static_cast<int32_t>(r.blocks.size()));
    r.blocks.clear();
    ++r.generation;
    r.num_computed = 0;
    r.state = PHOTON_REQ_PREEMPTED;
    s->waiting.push_front(id);
    ++b->num_preempted;
  }
  int64_t tokens = 0;
  for (int64_t id : s->running) {
    Request &r = s->reqs[id];
    const int64_t need = ceil_div(r.known(), bs) - static_cast<int64_t>(r.blocks.size());
    if (need > 0) {
      const size_t old = r.blocks.size();
      r.blocks.resize(old + static_cast<size_t>(need));
      if (photon_block_pool_alloc(s->pool, static_cast<int32_t>(need), r.blocks.data() + old) !=
          PHOTON_OK)
        return PHOTON_ERR_POOL_EXHAUSTED;  // not reachable: capacity checked above
    }
    tokens += r.known() - r.num_computed;
  }

  // ---- phase 2: admit waiting requests, first come first served
  while (!s->waiting.empty() && static_cast<int32_t>(s->running.size()) < s->cfg.max_running) {
    const int64_t id = s->waiting.front();
    Request &r = s->reqs[id];
    const int64_t new_tokens = r.known() - r.num_computed;
    const int64_t need = ceil_div(r.known(), bs);
    if (tokens + new_tokens > s->cfg.max_step_tokens) break;
    if (need > photon_block_pool_num_free(s->pool)) break;
    r.blocks.resize(static_cast<size_t>(need));
    if (photon_block_pool_alloc(s->pool, static_cast<int32_t>(need), r.blocks.data()) != PHOTON_OK)
      return PHOTON_ERR_POOL_EXHAUSTED;  // not reachable
    r.state = PHOTON_REQ_RUNNING;
    s->waiting.pop_front();
    s->running.push_back(id);
    tokens += new_tokens;
    ++b->num_admitted;
  }

  // ---- emit the batch: one row per running request, in admission order.
  // A row that holds the same request, with the same allocation (no
  // preemption in between), as in the previous batch written to this same
  // buffer only receives its new blocks; any other row is written whole
  // (entries past the request's blocks are -1).
  const int32_t W = s->cfg.max_blocks_per_seq;
  if (b->block_tables != s->last_tables) {
    s->row_id.assign(static_cast<size_t>(b->max_seqs), INT64_MIN);
    s->row_gen.assign(static_cast<size_t>(b->max_seqs), 0);
    s->row_len.assign(static_cast<size_t>(b->max_seqs), 0);
    s->last_tables = b->block_tables;
  }
  int32_t t = 0, max_ctx = 0;
  for (size_t i = 0; i < s->running.size(); ++i) {
    const Request &r = s->reqs[s->running[i]];
    b->request_ids[i] = r.id;
    b->num_new_tokens[i] = r.known() - r.num_computed;
    b->context_lens[i] = r.known();
    int32_t *row = b->block_tables + static_cast<int64_t>(i) * W;
    const int32_t nblk = static_cast<int32_t>(r.blocks.size());
    if (s->row_id[i] == r.id && s->row_gen[i] == r.generation && s->row_len[i] <= nblk) {
      for (int32_t j = s->row_len[i]; j < nblk; ++j) row[j] = r.blocks[j];
    } else {
      for (int32_t j = 0; j < W; ++j) row[j] = j < nblk ? r.blocks[j] : -1;
    }
    s->row_id[i] = r.id;
    s->row_gen[i] = r.generation;
    s->row_len[i] = nblk;
    for (int32_t p = r.num_computed; p < r.known(); ++p, ++t) {
      b->token_seq[t] = static_cast<int32_t>(i);
      b->positions[t] = p;
      b->slot_mapping[t] = static_cast<int64_t>(r.blocks[p / bs]) * bs + p % bs;
    }
    max_ctx = std::max(max_ctx, r.known());
  }
  b->num_seqs = static_cast<int32_t>(s->running.size());
  b->num_tokens = t;
  b->max_context_len = max_ctx;
  s->stepped = s->running;
  s->step_open = true;
  return PHOTON_OK;
}

int photon_scheduler_complete_step(photon_scheduler *s) {
  if (!s || !s->step_open) return PHOTON_ERR_INVALID_ARG;
  std::vector<int64_t> still;
  still.reserve(s->running.size());
  for (int64_t id : s->stepped) {
    Request &r = s->reqs[id];
    r.num_computed = r.known();
    r.num_generated += 1;
    if (r.num_generated >= r.max_new) {
      photon_block_pool_free(s->pool, r.blocks.data(), static_cast<int32_t>(r.blocks.size()));
      r.blocks.clear();
      r.state = PHOTON_REQ_FINISHED;
    } else {
      still.push_back(id);
    }
  }
  s->running = std::move(still);
  s->stepped.clear();
  s->step_open = false;
  return PHOTON_OK;
}

int photon_scheduler_request_state(const photon_scheduler *s, int64_t request_id, int32_t *state,
                                   int32_t *num_computed_tokens, int32_t *num_generated) {
  if (!s) return PHOTON_ERR_INVALID_ARG;
  auto it = s->reqs.find(request_id);
  if (it == s->reqs.end()) return PHOTON_ERR_INVALID_ARG;
  if (state) *state = it->second.state;
  if (num_computed_tokens) *num_computed_tokens = it->second.num_computed;
  if (num_generated) *num_generated = it->second.num_generated;
  return PHOTON_OK;
}

int photon_scheduler_counts(const photon_scheduler *s, int32_t *num_waiting, int32_t *num_running,
                            int32_t *num_finished) {
  if (!s) return PHOTON_ERR_INVALID_ARG;
  int32_t fin = 0;
  for (auto &kv : s->reqs) fin += kv.second.state == PHOTON_REQ_FINISHED;
  if (num_waiting) *num_waiting = static_cast<int32_t>(s->waiting.size());
  if (num_running) *num_running = static_cast<int32_t>(s->running.size());
  if (num_finished) *num_finished = fin;
  return PHOTON_OK;
}

}  // extern "C"
