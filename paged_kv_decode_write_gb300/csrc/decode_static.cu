// photon_paged_attention_decode_static: the decode step for callers that
// cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) at all:
// a plugin whose host application owns the whole device-memory budget and
// hands out no buffers, or a latency-critical serving loop where an
// allocation could synchronise the device and stall every other stream.
// Those callers still own q, the caches, the tables and `out`, but they have
// nowhere to put the split-K partials.  This entry point keeps them in a
// fixed scratch array compiled into the library instead of a caller-provided
// workspace, and otherwise runs exactly the kernels of
// photon_paged_attention_decode.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds PHOTON_STATIC_SCRATCH_BYTES of device memory until the
// process exits.  Host code only sees a stand-in symbol for it: its device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) on the first call made on that device, and cached.
#include <atomic>
#include <cstdint>

#include "internal.h"

namespace photon {
namespace {

constexpr int kMaxStaticDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[PHOTON_STATIC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device, or nullptr.
void *static_scratch_address() {
  static std::atomic<void *> addr[kMaxStaticDevices];  // races look it up twice
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStaticDevices) return nullptr;
  void *a = addr[dev].load(std::memory_order_relaxed);
  if (a == nullptr) {
    if (cudaGetSymbolAddress(&a, g_decode_scratch) != cudaSuccess) return nullptr;
    addr[dev].store(a, std::memory_order_relaxed);
  }
  return a;
}

}  // namespace
}  // namespace photon

extern "C" int photon_paged_attention_decode_static(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    const int32_t *context_lens, float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
    int32_t max_blocks_per_seq, int32_t max_context_len, int32_t partition_size,
    photon_dtype kv_dtype, photon_dtype out_dtype, photon_stream_t stream) {
  // the arguments first, so that a bad request gets its own status rather
  // than the size one
  const int rc = photon::check_decode_args(q, k_cache, v_cache, block_tables, context_lens, scale,
                                           out, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                           block_size, num_blocks, max_blocks_per_seq,
                                           max_context_len, partition_size, kv_dtype, out_dtype);
  if (rc != PHOTON_OK) return rc;
  const size_t need = photon_paged_attention_workspace_size(num_seqs, num_q_heads, head_dim,
                                                            max_context_len, partition_size);
  if (need > PHOTON_STATIC_SCRATCH_BYTES) return PHOTON_ERR_WORKSPACE;  // too large for the array
  void *ws = nullptr;
  if (need > 0 && num_seqs > 0) {
    ws = photon::static_scratch_address();
    if (ws == nullptr) return PHOTON_ERR_CUDA;
  }
  // Every partial the merge reads is written earlier in the same call, so
  // nothing left in the array by a previous call needs clearing.
  return photon_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       num_blocks, max_blocks_per_seq, max_context_len,
                                       partition_size, kv_dtype, out_dtype, ws, need, stream);
}
