// Ragged batch metadata on the host: the physical block pool and the
// per-step slot numbers / positions / context lengths a two-phase scheduler
// step hands to the kernels.
//
// PhotonInfer README, "Technical details > Paged attention" (block-level KV
// cache without fragmentation; per-sequence cache offsets) and
// "Technical details > Continuous batching scheduler" (running requests
// continue, waiting requests are admitted, num_computed_tokens marks where a
// request resumes).  Plain C++; no CUDA.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "photon.h"

struct photon_block_pool {
  std::vector<int32_t> free_list;  // top of the stack = next block handed out
  std::vector<uint8_t> in_use;     // 1 while a block is allocated
};

namespace {

// splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): a counter-based 64-bit generator.
uint64_t splitmix64(uint64_t &state) {
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Uniform integer in [0, n) by rejection (no modulo bias).
uint64_t uniform_below(uint64_t &state, uint64_t n) {
  const uint64_t limit = UINT64_MAX - UINT64_MAX % n;
  uint64_t r;
  do {
    r = splitmix64(state);
  } while (r >= limit);
  return r % n;
}

}  // namespace

extern "C" {

int photon_block_pool_create(int64_t num_blocks, uint64_t seed, photon_block_pool **out) {
  if (!out || num_blocks <= 0 || num_blocks > INT32_MAX) return PHOTON_ERR_INVALID_ARG;
  *out = nullptr;
  photon_block_pool *p = new (std::nothrow) photon_block_pool;
  if (!p) return PHOTON_ERR_INVALID_ARG;
  try {
    p->free_list.resize(static_cast<size_t>(num_blocks));
    p->in_use.assign(static_cast<size_t>(num_blocks), 0);
  } catch (...) {
    delete p;
    return PHOTON_ERR_INVALID_ARG;
  }
  for (int64_t i = 0; i < num_blocks; ++i) p->free_list[i] = static_cast<int32_t>(i);
  uint64_t st = seed;
  for (int64_t i = num_blocks - 1; i > 0; --i) {  // Fisher-Yates
    const int64_t j = static_cast<int64_t>(uniform_below(st, static_cast<uint64_t>(i + 1)));
    const int32_t t = p->free_list[i];
    p->free_list[i] = p->free_list[j];
    p->free_list[j] = t;
  }
  *out = p;
  return PHOTON_OK;
}

void photon_block_pool_destroy(photon_block_pool *pool) { delete pool; }

int64_t photon_block_pool_num_free(const photon_block_pool *pool) {
  return pool ? static_cast<int64_t>(pool->free_list.size()) : 0;
}

int photon_block_pool_alloc(photon_block_pool *pool, int32_t n, int32_t *ids_out) {
  if (!pool || n < 0 || (n > 0 && !ids_out)) return PHOTON_ERR_INVALID_ARG;
  if (static_cast<size_t>(n) > pool->free_list.size()) return PHOTON_ERR_POOL_EXHAUSTED;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = pool->free_list.back();
    pool->free_list.pop_back();
    pool->in_use[b] = 1;
    ids_out[i] = b;
  }
  return PHOTON_OK;
}

int photon_block_pool_free(photon_block_pool *pool, const int32_t *ids, int32_t n) {
  if (!pool || n < 0 || (n > 0 && !ids)) return PHOTON_ERR_INVALID_ARG;
  const int64_t nb = static_cast<int64_t>(pool->in_use.size());
  // validate everything first (including duplicates inside `ids`), then free
  std::vector<int32_t> seen;
  seen.reserve(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = ids[i];
    if (b < 0 || b >= nb || pool->in_use[b] != 1) {
      for (int32_t x : seen) pool->in_use[x] = 1;  // undo the provisional marks
      return PHOTON_ERR_INVALID_ARG;
    }
    pool->in_use[b] = 2;  // provisional mark catches a repeat within this call
    seen.push_back(b);
  }
  for (int32_t i = 0; i < n; ++i) {
    pool->in_use[ids[i]] = 0;
    pool->free_list.push_back(ids[i]);
  }
  return PHOTON_OK;
}

int photon_slot_mapping(const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                        const int32_t *token_seq, const int32_t *positions, int32_t num_tokens,
                        int32_t block_size, int64_t *slot_mapping) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_tokens < 0 || block_size <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!token_seq || !positions || !slot_mapping || !block_tables))
    return PHOTON_ERR_INVALID_ARG;
  for (int32_t t = 0; t < num_tokens; ++t)
    if (token_seq[t] < 0 || token_seq[t] >= num_seqs) return PHOTON_ERR_INVALID_ARG;
  for (int32_t t = 0; t < num_tokens; ++t) {
    const int32_t s = token_seq[t], p = positions[t];
    int64_t slot = -1;
    if (p >= 0 && p / block_size < max_blocks_per_seq) {
      const int32_t b = block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + p / block_size];
      if (b >= 0) slot = static_cast<int64_t>(b) * block_size + p % block_size;
    }
    slot_mapping[t] = slot;
  }
  return PHOTON_OK;
}

int photon_build_step_metadata(int32_t num_seqs, const int32_t *num_computed_tokens,
                               const int32_t *num_new_tokens, int32_t block_size,
                               int32_t *block_tables, int32_t max_blocks_per_seq,
                               photon_block_pool *pool, int32_t max_tokens, int32_t *token_seq,
                               int32_t *positions, int64_t *slot_mapping, int32_t *context_lens,
                               int32_t *num_tokens_out, int32_t *max_context_len_out) {
  if (num_seqs < 0 || block_size <= 0 || max_blocks_per_seq <= 0 || max_tokens < 0)
    return PHOTON_ERR_INVALID_ARG;
  if (!num_tokens_out || !max_context_len_out) return PHOTON_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!num_computed_tokens || !num_new_tokens || !block_tables || !context_lens))
    return PHOTON_ERR_INVALID_ARG;
  // pass 1: validate, count tokens and the blocks each row still needs
  int64_t total_tokens = 0, blocks_needed = 0;
  std::vector<int32_t> have(static_cast<size_t>(num_seqs), 0);
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int64_t c = num_computed_tokens[s], n = num_new_tokens[s];
    if (c < 0 || n < 0 || c + n > INT32_MAX) return PHOTON_ERR_INVALID_ARG;
    const int64_t need = (c + n + block_size - 1) / block_size;
    if (need > max_blocks_per_seq) return PHOTON_ERR_INVALID_ARG;
    const int32_t *row = block_tables + static_cast<int64_t>(s) * max_blocks_per_seq;
    int32_t h = 0;
    while (h < max_blocks_per_seq && row[h] >= 0) ++h;  // rows are filled left to right
    have[s] = h;
    if (need > h) blocks_needed += need - h;
    total_tokens += n;
  }
  if (total_tokens > max_tokens) return PHOTON_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!token_seq || !positions || !slot_mapping)) return PHOTON_ERR_INVALID_ARG;
  if (blocks_needed > 0) {
    if (!pool) return PHOTON_ERR_INVALID_ARG;
    if (blocks_needed > photon_block_pool_num_free(pool)) return PHOTON_ERR_POOL_EXHAUSTED;
  }
  // pass 2: grow rows, emit tokens
  int32_t t = 0, max_ctx = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t c = num_computed_tokens[s], n = num_new_tokens[s];
    int32_t *row = block_tables + static_cast<int64_t>(s) * max_blocks_per_seq;
    const int32_t need = static_cast<int32_t>((static_cast<int64_t>(c) + n + block_size - 1) / block_size);
    if (need > have[s]) {
      const int rc = photon_block_pool_alloc(pool, need - have[s], row + have[s]);
      if (rc != PHOTON_OK) return rc;  // cannot happen: capacity checked above
    }
    for (int32_t i = 0; i < n; ++i, ++t) {
      const int32_t p = c + i;
      token_seq[t] = s;
      positions[t] = p;
      slot_mapping[t] = static_cast<int64_t>(row[p / block_size]) * block_size + p % block_size;
    }
    context_lens[s] = c + n;
    if (c + n > max_ctx) max_ctx = c + n;
  }
  *num_tokens_out = t;
  *max_context_len_out = max_ctx;
  return PHOTON_OK;
}

}  // extern "C"
