// C ABI of the paged-KV decode library: argument validation, workspace
// sizing, and kernel dispatch.  Nothing here allocates device memory or
// synchronises a stream (photon_device_errors, a diagnostic, excepted).
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace photon {
namespace {

constexpr int kMaxDevices = 64;

// The library's sticky error word, one per device (a __device__ variable is
// instantiated in every context that loads the module).
__device__ unsigned int g_errors = 0;

unsigned int *error_word() {
  static std::atomic<unsigned int *> addr[kMaxDevices];  // races look it up twice
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int *a = addr[dev].load(std::memory_order_relaxed);
  if (a == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_errors) != cudaSuccess) return nullptr;
    a = static_cast<unsigned int *>(p);
    addr[dev].store(a, std::memory_order_relaxed);
  }
  return a;
}

// One warp waits on a phase nobody completes: the bounded wait must give up.
__global__ void selftest_wait_timeout_kernel(uint32_t budget, unsigned int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar, 0, budget));
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
    drain_async_copies();
  }
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool head_dim_ok(photon_dtype dt, int d) {
  if (dt == PHOTON_BF16) return d == 32 || d == 64 || d == 128 || d == 256;
  return d == 32 || d == 64 || d == 128;
}

bool group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PHOTON_OK : PHOTON_ERR_CUDA; }

struct Prepared {
  DecodeArgs args;
  WorkspaceLayout ws;
};

// Shared validation of the decode entry points.  Returns PHOTON_OK and fills
// `out`, or an error status with nothing launched.
int prepare_decode(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_tables, const int32_t *context_lens, float scale,
                   void *out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t block_size, int64_t num_blocks,
                   int32_t max_blocks_per_seq, int32_t max_context_len, int32_t partition_size,
                   photon_dtype kv_dtype, photon_dtype out_dtype, void *workspace,
                   size_t workspace_bytes, Prepared *prep, bool check_workspace = true) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || partition_size <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (kv_dtype != PHOTON_F32 && kv_dtype != PHOTON_BF16) return PHOTON_ERR_INVALID_ARG;
  if (out_dtype != PHOTON_F32 && out_dtype != PHOTON_BF16) return PHOTON_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PHOTON_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PHOTON_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PHOTON_ERR_UNSUPPORTED;
  if (partition_size % block_size != 0) return PHOTON_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_context_len)
    return PHOTON_ERR_INVALID_ARG;
  if (!head_dim_ok(kv_dtype, head_dim) || !group_ok(num_q_heads / num_kv_heads))
    return PHOTON_ERR_UNSUPPORTED;
  if (num_blocks > INT32_MAX) return PHOTON_ERR_UNSUPPORTED;  // block ids are int32
  WorkspaceLayout ws = workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                                        partition_size);
  const int64_t items = static_cast<int64_t>(num_seqs) * ws.max_partitions * num_kv_heads;
  if (items > INT32_MAX / 2) return PHOTON_ERR_UNSUPPORTED;
  if (num_seqs > 0) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
      return PHOTON_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
      return PHOTON_ERR_INVALID_ARG;
    if (check_workspace && ws.total > 0 &&
        (!workspace || !aligned(workspace, 16) || workspace_bytes < ws.total))
      return PHOTON_ERR_WORKSPACE;
  }
  DecodeArgs &a = prep->args;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  char *w = static_cast<char *>(workspace);
  a.m_part = ws.total ? reinterpret_cast<float *>(w + ws.m_off) : nullptr;
  a.l_part = ws.total ? reinterpret_cast<float *>(w + ws.l_off) : nullptr;
  a.o_part = ws.total ? reinterpret_cast<float *>(w + ws.o_off) : nullptr;
  a.seg_count = ws.total ? reinterpret_cast<int32_t *>(w + ws.c_off) : nullptr;
  a.ctl = ws.total ? reinterpret_cast<DecodeCtl *>(w + ws.x_off) : nullptr;
  a.num_blocks = num_blocks;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // log2(e)
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.ctx_cap = max_context_len;
  a.partition_size = partition_size;
  a.max_partitions = ws.slots;
  a.balanced = 0;
  a.out_bf16 = out_dtype == PHOTON_BF16;
  a.row_of_seq = nullptr;
  a.query_positions = nullptr;
  a.num_table_rows = num_seqs;
  prep->ws = ws;
  return PHOTON_OK;
}

int launch_partial(const Prepared &p, photon_dtype kv_dtype, cudaStream_t st) {
  unsigned int *err = error_word();
  if (!err) return PHOTON_ERR_CUDA;
  return cuda_status(kv_dtype == PHOTON_BF16 ? launch_decode_partial_bf16(p.args, err, st)
                                             : launch_decode_partial_f32(p.args, err, st));
}

}  // namespace

WorkspaceLayout workspace_layout(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t partition_size) {
  WorkspaceLayout w{};
  const int32_t P = (max_context_len <= 0 || partition_size <= 0)
                        ? 1
                        : (max_context_len + partition_size - 1) / partition_size;
  w.max_partitions = P;
  w.slots = P;
  if (P <= 1 || num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0) return w;
  w.slots = P + 1;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  const size_t n = rows * w.slots;
  w.m_off = 0;
  w.l_off = align256(n * sizeof(float));
  w.o_off = 2 * align256(n * sizeof(float));
  w.c_off = w.o_off + align256(n * head_dim * sizeof(float));
  w.x_off = w.c_off + (rows + 1 + 3) / 4 * 16;  // the counts, rounded up to 16 bytes
  w.total = w.c_off + align256(w.x_off - w.c_off + sizeof(DecodeCtl));
  return w;
}

int check_decode_args(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, float scale,
                      void *out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int64_t num_blocks,
                      int32_t max_blocks_per_seq, int32_t max_context_len,
                      int32_t partition_size, photon_dtype kv_dtype, photon_dtype out_dtype) {
  Prepared p{};
  return prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                        max_blocks_per_seq, max_context_len, partition_size, kv_dtype, out_dtype,
                        nullptr, 0, &p, /*check_workspace=*/false);
}

int device_sm_count() {
  static std::atomic<int> count[kMaxDevices];  // 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int c = count[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 1;
    count[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace photon

using namespace photon;

namespace photon {
namespace {

int kv_cache_write_impl(void *q, const int32_t *q_positions, int32_t num_q_tokens,
                        int32_t num_q_heads, const void *k, const void *v,
                        const int32_t *positions, const int64_t *slot_mapping, void *k_cache,
                        void *v_cache, int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t num_blocks, photon_dtype kv_dtype,
                        float rope_theta, photon_rope rope_style, photon_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
      num_q_tokens < 0 || (q && num_q_heads <= 0))
    return PHOTON_ERR_INVALID_ARG;
  if (kv_dtype != PHOTON_F32 && kv_dtype != PHOTON_BF16) return PHOTON_ERR_INVALID_ARG;
  if (rope_style != PHOTON_ROPE_NEOX && rope_style != PHOTON_ROPE_GPTJ &&
      rope_style != PHOTON_ROPE_NONE)
    return PHOTON_ERR_INVALID_ARG;
  if (rope_style != PHOTON_ROPE_NONE && !(std::isfinite(rope_theta) && rope_theta > 0.f))
    return PHOTON_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PHOTON_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return PHOTON_ERR_UNSUPPORTED;
  if (num_blocks > INT64_MAX / (static_cast<int64_t>(num_kv_heads) * block_size * head_dim))
    return PHOTON_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) + num_q_tokens > INT32_MAX) return PHOTON_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!k || !v || !positions || !slot_mapping || !k_cache || !v_cache)
      return PHOTON_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(positions, 4) || !aligned(slot_mapping, 8))
      return PHOTON_ERR_INVALID_ARG;
  }
  if (q && num_q_tokens > 0 && (!q_positions || !aligned(q, 16) || !aligned(q_positions, 4)))
    return PHOTON_ERR_INVALID_ARG;
  if (num_tokens == 0 && (!q || num_q_tokens == 0)) return PHOTON_OK;
  WriteArgs a{};
  a.k = k;
  a.v = v;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.q = q;
  a.q_positions = q_positions;
  a.num_q_tokens = q ? num_q_tokens : 0;
  a.num_q_heads = num_q_heads;
  a.num_slots = num_blocks * block_size;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.rope_style = rope_style;
  for (int i = 0; i < head_dim / 2; ++i)
    a.inv_freq[i] = std::pow(static_cast<double>(rope_theta), -2.0 * i / head_dim);
  unsigned int *err = error_word();
  if (!err) return PHOTON_ERR_CUDA;
  return cuda_status(launch_kv_cache_write(a, kv_dtype, err, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace photon


extern "C" {

const char *photon_status_string(int status) {
  switch (status) {
    case PHOTON_OK: return "ok";
    case PHOTON_ERR_INVALID_ARG: return "invalid argument";
    case PHOTON_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PHOTON_ERR_WORKSPACE: return "workspace missing or too small";
    case PHOTON_ERR_CUDA: return "CUDA error";
    case PHOTON_ERR_POOL_EXHAUSTED: return "block pool exhausted";
    default: return "unknown status";
  }
}

int photon_version(void) { return 100; }

int photon_kv_cache_write(const void *k, const void *v, const int32_t *positions,
                          const int64_t *slot_mapping, void *k_cache, void *v_cache,
                          int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int64_t num_blocks, photon_dtype kv_dtype,
                          float rope_theta, photon_rope rope_style, photon_stream_t stream) {
  return photon::kv_cache_write_impl(nullptr, nullptr, 0, 0, k, v, positions, slot_mapping, k_cache,
                             v_cache, num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
                             kv_dtype, rope_theta, rope_style, stream);
}

int photon_rope_q_kv_cache_write(void *q, const int32_t *q_positions, int32_t num_q_tokens,
                                 int32_t num_q_heads, const void *k, const void *v,
                                 const int32_t *positions, const int64_t *slot_mapping,
                                 void *k_cache, void *v_cache, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, photon_dtype kv_dtype, float rope_theta,
                                 photon_rope rope_style, photon_stream_t stream) {
  if (!q && num_q_tokens > 0) return PHOTON_ERR_INVALID_ARG;
  return photon::kv_cache_write_impl(q, q_positions, num_q_tokens, num_q_heads, k, v, positions,
                             slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim,
                             block_size, num_blocks, kv_dtype, rope_theta, rope_style, stream);
}

size_t photon_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                             int32_t head_dim, int32_t max_context_len,
                                             int32_t partition_size) {
  return workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size).total;
}

int photon_paged_attention_partial(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, int32_t max_blocks_per_seq,
                                   int32_t max_context_len, int32_t partition_size,
                                   photon_dtype kv_dtype, photon_dtype out_dtype, void *workspace,
                                   size_t workspace_bytes, photon_stream_t stream) {
  Prepared p{};
  int rc = prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          max_blocks_per_seq, max_context_len, partition_size, kv_dtype,
                          out_dtype, workspace, workspace_bytes, &p);
  if (rc != PHOTON_OK || num_seqs == 0) return rc;
  return launch_partial(p, kv_dtype, reinterpret_cast<cudaStream_t>(stream));
}

int photon_paged_attention_reduce(const int32_t *context_lens, void *out, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t head_dim, int32_t max_context_len,
                                  int32_t partition_size, photon_dtype out_dtype, void *workspace,
                                  size_t workspace_bytes, photon_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || partition_size <= 0 ||
      partition_size % kBlockSize != 0)
    return PHOTON_ERR_INVALID_ARG;
  if (out_dtype != PHOTON_F32 && out_dtype != PHOTON_BF16) return PHOTON_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return PHOTON_ERR_UNSUPPORTED;
  WorkspaceLayout ws = workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                                        partition_size);
  if (num_seqs == 0 || ws.total == 0) return PHOTON_OK;  // nothing was split
  if (!context_lens || !out) return PHOTON_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < ws.total)
    return PHOTON_ERR_WORKSPACE;
  DecodeArgs a{};
  char *w = static_cast<char *>(workspace);
  a.context_lens = context_lens;
  a.out = out;
  a.m_part = reinterpret_cast<float *>(w + ws.m_off);
  a.l_part = reinterpret_cast<float *>(w + ws.l_off);
  a.o_part = reinterpret_cast<float *>(w + ws.o_off);
  a.seg_count = reinterpret_cast<int32_t *>(w + ws.c_off);
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.head_dim = head_dim;
  a.ctx_cap = max_context_len;
  a.partition_size = partition_size;
  a.max_partitions = ws.slots;
  a.out_bf16 = out_dtype == PHOTON_BF16;
  return cuda_status(launch_decode_reduce(a, reinterpret_cast<cudaStream_t>(stream)));
}

int photon_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, int32_t max_blocks_per_seq,
                                  int32_t max_context_len, int32_t partition_size,
                                  photon_dtype kv_dtype, photon_dtype out_dtype, void *workspace,
                                  size_t workspace_bytes, photon_stream_t stream) {
  Prepared p{};
  int rc = prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          max_blocks_per_seq, max_context_len, partition_size, kv_dtype,
                          out_dtype, workspace, workspace_bytes, &p);
  if (rc != PHOTON_OK || num_seqs == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_partial(p, kv_dtype, st);
  if (rc != PHOTON_OK || p.ws.total == 0) return rc;
  return cuda_status(launch_decode_reduce(p.args, st));
}

int photon_kv_cache_write_fp8(const void *k, const void *v, const int32_t *positions,
                              const int64_t *slot_mapping, void *k_cache, void *v_cache,
                              const float *k_scale, const float *v_scale, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, photon_dtype in_dtype, float rope_theta,
                              photon_rope rope_style, photon_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
    return PHOTON_ERR_INVALID_ARG;
  if (in_dtype != PHOTON_F32 && in_dtype != PHOTON_BF16) return PHOTON_ERR_INVALID_ARG;
  if (rope_style != PHOTON_ROPE_NEOX && rope_style != PHOTON_ROPE_GPTJ &&
      rope_style != PHOTON_ROPE_NONE)
    return PHOTON_ERR_INVALID_ARG;
  if (rope_style != PHOTON_ROPE_NONE && !(std::isfinite(rope_theta) && rope_theta > 0.f))
    return PHOTON_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PHOTON_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return PHOTON_ERR_UNSUPPORTED;
  if (num_blocks > INT64_MAX / (static_cast<int64_t>(num_kv_heads) * block_size * head_dim))
    return PHOTON_ERR_INVALID_ARG;
  if (num_kv_heads > 64) return PHOTON_ERR_UNSUPPORTED;  // per-head scales staged on chip
  if (num_tokens == 0) return PHOTON_OK;
  if (!k || !v || !positions || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PHOTON_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(positions, 4) || !aligned(slot_mapping, 8) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4))
    return PHOTON_ERR_INVALID_ARG;
  WriteArgs a{};
  a.k = k;
  a.v = v;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_slots = num_blocks * block_size;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.rope_style = rope_style;
  for (int i = 0; i < head_dim / 2; ++i)
    a.inv_freq[i] = std::pow(static_cast<double>(rope_theta), -2.0 * i / head_dim);
  unsigned int *err = error_word();
  if (!err) return PHOTON_ERR_CUDA;
  return cuda_status(launch_kv_cache_write_fp8(a, in_dtype, k_scale, v_scale, err,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace photon {
namespace {

// The FP8 decode: the partial kernel, then (merge) the log-sum-exp merge.
int decode_fp8_impl(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                    const float *v_scale, const int32_t *block_tables, const int32_t *context_lens,
                    float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                    int32_t max_blocks_per_seq, int32_t max_context_len, int32_t partition_size,
                    photon_dtype out_dtype, void *workspace, size_t workspace_bytes,
                    photon_stream_t stream, bool merge) {
  Prepared p{};
  int rc = prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          max_blocks_per_seq, max_context_len, partition_size, PHOTON_BF16,
                          out_dtype, workspace, workspace_bytes, &p);
  if (rc != PHOTON_OK) return rc;
  if (head_dim != 64 && head_dim != 128) return PHOTON_ERR_UNSUPPORTED;
  if (num_seqs > 0 && (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4)))
    return PHOTON_ERR_INVALID_ARG;
  if (num_seqs == 0) return PHOTON_OK;
  unsigned int *err = error_word();
  if (!err) return PHOTON_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = cuda_status(launch_decode_partial_fp8(p.args, k_scale, v_scale, err, st));
  if (rc != PHOTON_OK || p.ws.total == 0 || !merge) return rc;
  return cuda_status(launch_decode_reduce(p.args, st));
}

}  // namespace
}  // namespace photon

extern "C" {

int photon_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, const int32_t *context_lens,
                                      float scale, void *out, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks,
                                      int32_t max_blocks_per_seq, int32_t max_context_len,
                                      int32_t partition_size, photon_dtype out_dtype,
                                      void *workspace, size_t workspace_bytes,
                                      photon_stream_t stream) {
  return photon::decode_fp8_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                 scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, max_context_len,
                                 partition_size, out_dtype, workspace, workspace_bytes, stream,
                                 true);
}

int photon_paged_attention_partial_fp8(const void *q, const void *k_cache, const void *v_cache,
                                       const float *k_scale, const float *v_scale,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       float scale, void *out, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int32_t max_blocks_per_seq, int32_t max_context_len,
                                       int32_t partition_size, photon_dtype out_dtype,
                                       void *workspace, size_t workspace_bytes,
                                       photon_stream_t stream) {
  return photon::decode_fp8_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                 scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, max_context_len,
                                 partition_size, out_dtype, workspace, workspace_bytes, stream,
                                 false);
}

int photon_paged_attention_prefill(const void *q, const int32_t *token_seq,
                                   const int32_t *positions, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables, float scale,
                                   void *out, int32_t num_tokens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_blocks,
                                   int32_t max_blocks_per_seq, int32_t max_position,
                                   int32_t partition_size, photon_dtype kv_dtype,
                                   photon_dtype out_dtype, void *workspace,
                                   size_t workspace_bytes, photon_stream_t stream) {
  if (num_seqs < 0 || max_position < 0 || max_position == INT32_MAX) return PHOTON_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!token_seq || !positions || !aligned(token_seq, 4) || !aligned(positions, 4)))
    return PHOTON_ERR_INVALID_ARG;
  // every query token is a sequence: context = position + 1, table row = its sequence
  Prepared p{};
  int rc = prepare_decode(q, k_cache, v_cache, block_tables, positions, scale, out, num_tokens,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          max_blocks_per_seq, max_position + 1, partition_size, kv_dtype,
                          out_dtype, workspace, workspace_bytes, &p);
  if (rc != PHOTON_OK || num_tokens == 0) return rc;
  p.args.row_of_seq = token_seq;
  p.args.query_positions = positions;
  p.args.num_table_rows = num_seqs;
  p.args.seg_count = nullptr;  // the merge counts each token's partitions
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (prefill_tiled_supported(p.args, kv_dtype)) {
    unsigned int *err = error_word();
    if (!err) return PHOTON_ERR_CUDA;
    rc = cuda_status(prefill_tc_preferred(p.args) ? launch_prefill_tc(&p.args, err, st)
                                                  : launch_prefill_tiled(&p.args, err, st));
  } else {
    rc = launch_partial(p, kv_dtype, st);  // one decode query per token
  }
  if (rc != PHOTON_OK || p.ws.total == 0) return rc;
  // every token's context fits one (possibly coarsened) partition: the
  // partial kernel wrote all outputs, nothing to merge
  if (static_cast<int64_t>(max_position) + 1 <= p.args.partition_size) return rc;
  return cuda_status(launch_decode_reduce(p.args, st));
}

int photon_selftest_wait_timeout(uint32_t budget_cycles, photon_stream_t stream) {
  if (budget_cycles == 0) return PHOTON_ERR_INVALID_ARG;
  unsigned int *err = error_word();
  if (!err) return PHOTON_ERR_CUDA;
  selftest_wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_cycles,
                                                                                      err);
  return cuda_status(cudaGetLastError());
}

int photon_device_errors(uint32_t *flags_out, int clear) {
  if (!flags_out) return PHOTON_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return PHOTON_ERR_CUDA;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_errors, sizeof v);
  if (e != cudaSuccess) return PHOTON_ERR_CUDA;
  *flags_out = v;
  if (clear) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_errors, &z, sizeof z);
    if (e != cudaSuccess) return PHOTON_ERR_CUDA;
  }
  return PHOTON_OK;
}

}  // extern "C"
