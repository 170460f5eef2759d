// Host-side declarations shared by the C ABI (photon_abi.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "photon.h"

namespace photon {

constexpr int kBlockSize = 16;     // tokens per physical KV block
constexpr int kMaxRopePairs = 128; // head_dim <= 256

struct WriteArgs {
  const void *k;
  const void *v;
  const int32_t *positions;
  const int64_t *slot_mapping;
  void *k_cache;
  void *v_cache;
  void *q;                    // optional: rows rotated in place by the same launch
  const int32_t *q_positions;
  int32_t num_q_tokens;
  int32_t num_q_heads;
  int64_t num_slots;  // num_blocks * block_size
  int32_t num_tokens;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t rope_style;
  double inv_freq[kMaxRopePairs];  // theta^(-2i/d), fp64, filled on the host
};

// Control block of a decode workspace (16 bytes, 8-byte aligned) for the
// tensor-core decode's dynamic item order: two counters, each a 64-bit word
// whose high 40 bits carry kCtlTag while a launch uses it and whose low 24
// bits count.  Between launches both words are 0.  A launch's first thread
// writes kCtlTag to both; an atomic add whose returned word lacks the tag
// came before that and is lost (its issuer tries again); the last warp to
// leave writes 0 to both.  A fresh (uninitialised) workspace holds the tag
// only by a 2^-40 chance.
struct DecodeCtl {
  unsigned long long next;  // items claimed after the warps' first ones
  unsigned long long done;  // warps that have left
};
constexpr int kCtlCountBits = 24;
constexpr unsigned long long kCtlTag = 0x9e3779b97full << kCtlCountBits;

struct DecodeArgs {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_tables;
  const int32_t *context_lens;
  void *out;
  float *m_part;  // [B][H_q][P_max]
  float *l_part;  // [B][H_q][P_max]
  float *o_part;  // [B][H_q][P_max][d]
  // Decode with a workspace: [B * H_q + 1] words.  Word B * H_q is the mode
  // of the last partial launch (0: fixed partitions, 1: page-balanced
  // pieces), written by its first thread; in mode 1 word r holds the number
  // of pieces of (sequence, query head) row r (1: the partial kernel wrote
  // the row itself).  The merge reads them.  NULL for prefill, whose merge
  // counts the partitions of the query's context.
  int32_t *seg_count;
  // Decode with a workspace: its control block (see DecodeCtl); NULL for
  // prefill and for workspace-free calls (items then go to the warps in a
  // fixed order).
  DecodeCtl *ctl;
  int64_t num_blocks;
  float scale_log2;  // scale * log2(e): scores are kept in base-2 units
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t max_blocks_per_seq;
  int32_t ctx_cap;  // min(max_context_len, max_blocks_per_seq * block_size)
  int32_t partition_size;
  int32_t max_partitions;  // pieces per row in the workspace (the row stride of the partials)
  // Tensor-core decode: 1 = page-balanced pieces (each warp of the grid one
  // equal run of the page stream, see walker_start), 0 = fixed partitions of
  // partition_size tokens.  Set by their launchers.
  int32_t balanced;
  int32_t out_bf16;
  // Prefill: every query token is a sequence of its own whose context is its
  // position + 1 and whose block-table row is row_of_seq[token] (both NULL
  // for decode, where sequence s uses row s and context_lens[s]).
  const int32_t *row_of_seq;
  const int32_t *query_positions;
  int32_t num_table_rows;
  // L2 lookahead of the tensor-core kernels, in pages (0 = off); set by
  // their launchers.
  int32_t l2_lookahead;
};

// Workspace carve-up for given sizes; all offsets 256-B aligned.
struct WorkspaceLayout {
  size_t m_off, l_off, o_off, c_off, x_off, total;  // x_off: the DecodeCtl
  int32_t max_partitions;  // partitions of partition_size tokens in max_context_len
  int32_t slots;           // pieces per row: max_partitions + 1 (a balanced run may split one)
};
WorkspaceLayout workspace_layout(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t partition_size);

// `err` is the device address of the library's sticky error word.
cudaError_t launch_kv_cache_write(const WriteArgs &a, photon_dtype dt, unsigned int *err,
                                  cudaStream_t st);
cudaError_t launch_decode_partial_bf16(const DecodeArgs &a, unsigned int *err, cudaStream_t st);
cudaError_t launch_decode_partial_f32(const DecodeArgs &a, unsigned int *err, cudaStream_t st);
cudaError_t launch_decode_reduce(const DecodeArgs &a, cudaStream_t st);
// Tiled tensor-core prefill (bf16 pools, head_dim 64/128, G in {1,2,4,8});
// DecodeArgs as for the per-token prefill (row_of_seq, query_positions).  It
// may coarsen a->partition_size (to a multiple of it); the merge that follows
// must use the updated value.
bool prefill_tiled_supported(const DecodeArgs &a, photon_dtype kv_dtype);
cudaError_t launch_prefill_tiled(DecodeArgs *a, unsigned int *err, cudaStream_t st);
// Prefill on tcgen05 / TMEM (same shapes as the tiled kernel): preferred when
// its 128-row tiles alone give every SM a work item.  Writes every output row
// (sets a->partition_size so that no merge follows).
bool prefill_tc_preferred(const DecodeArgs &a);
cudaError_t launch_prefill_tc(DecodeArgs *a, unsigned int *err, cudaStream_t st);
cudaError_t launch_kv_cache_write_fp8(const WriteArgs &a, photon_dtype in_dt, const float *k_scale,
                                      const float *v_scale, unsigned int *err, cudaStream_t st);
cudaError_t launch_decode_partial_fp8(const DecodeArgs &a, const float *k_scale,
                                      const float *v_scale, unsigned int *err, cudaStream_t st);

// Every host-side check of photon_paged_attention_decode except the workspace
// one: PHOTON_OK or the status that call would return, nothing launched.
int check_decode_args(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens, float scale,
                      void *out, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int64_t num_blocks,
                      int32_t max_blocks_per_seq, int32_t max_context_len,
                      int32_t partition_size, photon_dtype kv_dtype, photon_dtype out_dtype);

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();

}  // namespace photon
