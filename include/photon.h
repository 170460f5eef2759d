/*
 * photon.h -- C ABI of the GB300 (sm_103a) paged-KV decode library.
 *
 * One decode step of a continuous-batching LLM engine over a block-level
 * ("paged") KV cache, as the PhotonInfer README describes it:
 *   - "Technical details > Paged attention": the KV cache is allocated in
 *     fixed-size physical blocks with no fragmentation; each sequence keeps
 *     its own cache offsets (a block table); one batched kernel writes K/V
 *     for many sequences.
 *   - "Key features > GPU-optimised kernels": batched paged attention,
 *     batched RoPE fused into a kernel, numerically stable attention softmax.
 *   - "Technical details > Continuous batching scheduler": a two-phase
 *     scheduler step tracks num_computed_tokens per request; the metadata
 *     calls below turn that state into the per-token slot numbers and
 *     per-sequence context lengths the kernels consume.
 *   - "Key features > Modern C++20 architecture": errors are returned as
 *     explicit status values (the README's Result type), and every buffer is
 *     a non-owning view (its std::span, zero-copy design).
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership.  Every pointer is a view of caller-owned memory.  The library
 *   never allocates, frees, copies or retains a caller buffer, and never
 *   synchronises a stream on the kernel calls.  "device" pointers are CUDA
 *   device (or managed) memory on the current device; "host" pointers are
 *   ordinary host memory.
 * Streams.  photon_stream_t is a cudaStream_t (0 = legacy default stream).
 *   Kernel calls only enqueue work on it and return.  The kernels use
 *   programmatic dependent launch among themselves: a decode kernel may
 *   start while this library's preceding kernel on the stream is still
 *   running and read the batch's metadata (context lengths, block tables,
 *   prefill positions and token rows) early, before it waits for that kernel
 *   and touches anything else.  No kernel of the library writes that
 *   metadata, and any other kernel on the stream completes before the next
 *   one of the library starts, so stream order holds for every input.
 * Errors.  Every call returns a photon_status.  Arguments the host can check
 *   are checked before anything is launched (PHOTON_ERR_INVALID_ARG /
 *   PHOTON_ERR_UNSUPPORTED / PHOTON_ERR_WORKSPACE); a failed launch returns
 *   PHOTON_ERR_CUDA.  Device-resident metadata (slot numbers, block ids,
 *   context lengths) is checked inside the kernels: an out-of-range value is
 *   never dereferenced -- the access is skipped and a sticky bit is set,
 *   readable with photon_device_errors().  No kernel traps or waits without
 *   a bound.
 *
 * KV cache layout (one pool each for K and V):
 *   cache[num_blocks][num_kv_heads][block_size][head_dim], row-major, so
 *   element (b, h, o, e) sits at ((b*num_kv_heads + h)*block_size + o)*head_dim + e.
 *   A token at position p of sequence s lives in block block_tables[s][p/bs]
 *   at offset p % bs; its slot number is block*bs + offset.
 *
 * Supported shapes: head_dim in {32, 64, 128, 256}; block_size 16;
 *   num_q_heads / num_kv_heads in {1, 2, 4, 8}; storage type fp32 or bf16.
 */
#ifndef PHOTON_H
#define PHOTON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *photon_stream_t; /* == cudaStream_t */

typedef enum {
  PHOTON_OK = 0,
  PHOTON_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned buffer   */
  PHOTON_ERR_UNSUPPORTED = -2, /* valid request outside the compiled shapes   */
  PHOTON_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required  */
  PHOTON_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed        */
  PHOTON_ERR_POOL_EXHAUSTED = -5 /* block pool has fewer free blocks than asked */
} photon_status;

typedef enum { PHOTON_F32 = 0, PHOTON_BF16 = 1 } photon_dtype;

typedef enum {
  PHOTON_ROPE_NEOX = 0, /* pairs (i, i + d/2): "rotate half"      */
  PHOTON_ROPE_GPTJ = 1, /* pairs (2i, 2i + 1): interleaved        */
  PHOTON_ROPE_NONE = 2  /* no rotation: K is copied like V        */
} photon_rope;

/* Sticky device-side error bits (photon_device_errors). */
#define PHOTON_DEVERR_SLOT_RANGE 0x1u    /* a slot_mapping entry >= num_blocks*block_size: not written */
#define PHOTON_DEVERR_BLOCK_RANGE 0x2u   /* a block_tables entry outside [0, num_blocks): page skipped */
#define PHOTON_DEVERR_CONTEXT_RANGE 0x4u /* a context length above max_context_len or the table width: clamped */
#define PHOTON_DEVERR_WAIT_TIMEOUT 0x8u  /* a bounded wait on a page copy gave up: item abandoned */

/* Human-readable name of a status value (static string, never NULL). */
const char *photon_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int photon_version(void);

/*
 * photon_kv_cache_write -- the batched cache write ("one kernel writes K/V for
 * many sequences"), with RoPE fused in ("batched RoPE").
 *
 * For every token t < num_tokens with slot = slot_mapping[t] >= 0 and every
 * KV head h:
 *   k_cache[slot / bs][h][slot % bs][:] = round(RoPE(k[t][h][:], positions[t]))
 *   v_cache[slot / bs][h][slot % bs][:] = v[t][h][:]        (bit copy)
 * RoPE rotates pair (x_a, x_b) by the angle positions[t] * theta^(-2i/d)
 * (pair i of rope_style) using the fp64 sine and cosine of the angle; a bf16
 * cache stores the exact rotated value rounded once to nearest-even, an fp32
 * cache the fp64 rotation rounded once (within one unit in the last place).
 *
 *   k, v          device, [num_tokens][num_kv_heads][head_dim], kv_dtype, 16-B aligned
 *   positions     device int32 [num_tokens], >= 0
 *   slot_mapping  device int64 [num_tokens]; -1 = skip the token
 *   k_cache, v_cache  device, pool layout above, kv_dtype, 16-B aligned
 *   rope_theta    > 0 (ignored for PHOTON_ROPE_NONE)
 * Slots must be distinct (two tokens writing one slot race).  A slot outside
 * the pool is not written and sets PHOTON_DEVERR_SLOT_RANGE.
 */
int photon_kv_cache_write(const void *k, const void *v, const int32_t *positions,
                          const int64_t *slot_mapping, void *k_cache, void *v_cache,
                          int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int64_t num_blocks, photon_dtype kv_dtype,
                          float rope_theta, photon_rope rope_style, photon_stream_t stream);

/*
 * photon_rope_q_kv_cache_write -- photon_kv_cache_write plus the rotation of
 * this step's query rows, in the same launch ("batched RoPE" fused with the
 * batched cache write; the decode call then takes the rotated q).
 *
 *   q            device [num_q_tokens][num_q_heads][head_dim], kv_dtype,
 *                16-B aligned; rotated IN PLACE with RoPE at q_positions[i]
 *                (same angles, rounding and style as K)
 *   q_positions  device int32 [num_q_tokens], >= 0
 * All other arguments and behaviour as photon_kv_cache_write.  q may be NULL
 * only when num_q_tokens is 0.
 */
int photon_rope_q_kv_cache_write(void *q, const int32_t *q_positions, int32_t num_q_tokens,
                                 int32_t num_q_heads, const void *k, const void *v,
                                 const int32_t *positions, const int64_t *slot_mapping,
                                 void *k_cache, void *v_cache, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, photon_dtype kv_dtype, float rope_theta,
                                 photon_rope rope_style, photon_stream_t stream);

/*
 * Bytes of device workspace photon_paged_attention_decode needs (0 when no
 * sequence can span more than one partition).  Holds the split-K partial
 * results: for every (sequence, query head) P + 1 slots, P = the partitions
 * of partition_size tokens in max_context_len (one more because the FP8
 * decode's page-balanced pieces may cut a sequence once more than its
 * partitions), each the running maximum and exponential sum (fp32) and the
 * unnormalised output (fp32 x d); per (sequence, query head) the number
 * of pieces the partial kernel wrote (int32), which the merge reads; and a
 * 16-byte control block through which the tensor-core decode's warps claim
 * work items in dynamic order.  The block needs no initialisation: a call
 * marks it in use at its start and leaves it zeroed.  Calls that may run at
 * the same time need separate workspaces.
 */
size_t photon_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                             int32_t head_dim, int32_t max_context_len,
                                             int32_t partition_size);

/*
 * photon_paged_attention_decode -- batched paged attention for one query
 * token per sequence ("batched paged attention" over the block-level cache),
 * with grouped KV heads, a numerically stable online softmax and a split-K
 * partition of the context followed by a log-sum-exp merge.
 *
 * For sequence s (ctx = context_lens[s]) and query head g, with KV head
 * h = g / (num_q_heads / num_kv_heads):
 *   out[s][g][:] = sum_{j < ctx} softmax_j(scale * <q[s][g][:], K_s[h][j][:]>) * V_s[h][j][:]
 * where K_s / V_s are read through block_tables[s].  The context is cut into
 * partitions of partition_size tokens; each (sequence, KV head, partition)
 * yields partial (max, sum, output) triples that a second kernel merges.
 * Sequences with one partition are written directly.  ctx <= 0 gives a zero
 * row.  q is expected already rotated.
 *
 *   q             device [num_seqs][num_q_heads][head_dim], kv_dtype, 16-B aligned
 *   k_cache, v_cache  device, pool layout above, kv_dtype, 16-B aligned
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens  device int32 [num_seqs], each <= max_context_len
 *   out           device [num_seqs][num_q_heads][head_dim], out_dtype, 16-B aligned
 *   max_context_len  host-known upper bound of context_lens (sizes the grid
 *                 and workspace; no device read)
 *   partition_size  tokens per split-K partition, a positive multiple of block_size
 *   workspace     device, >= photon_paged_attention_workspace_size(...) bytes,
 *                 256-B aligned; may be NULL when that size is 0
 */
int photon_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, int32_t max_blocks_per_seq,
                                  int32_t max_context_len, int32_t partition_size,
                                  photon_dtype kv_dtype, photon_dtype out_dtype, void *workspace,
                                  size_t workspace_bytes, photon_stream_t stream);

/*
 * The two halves of photon_paged_attention_decode, for callers that schedule
 * or time them separately.  Called back to back on one stream with identical
 * arguments they do exactly what photon_paged_attention_decode does.
 *   _partial: per-(sequence, KV head, partition) attention; writes `out` for
 *             single-partition sequences and partials to the workspace.
 *   _reduce:  log-sum-exp merge of the partials into `out`, and zero rows for
 *             empty contexts.
 */
int photon_paged_attention_partial(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   float scale, void *out, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, int32_t max_blocks_per_seq,
                                   int32_t max_context_len, int32_t partition_size,
                                   photon_dtype kv_dtype, photon_dtype out_dtype, void *workspace,
                                   size_t workspace_bytes, photon_stream_t stream);
int photon_paged_attention_reduce(const int32_t *context_lens, void *out, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t head_dim, int32_t max_context_len,
                                  int32_t partition_size, photon_dtype out_dtype, void *workspace,
                                  size_t workspace_bytes, photon_stream_t stream);

/* Bytes of the scratch array that photon_paged_attention_decode_static uses
 * in place of a workspace (32 MiB, held on every device that loads the
 * library until the process exits). */
#define PHOTON_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * photon_paged_attention_decode_static -- photon_paged_attention_decode for
 * callers that cannot allocate device memory.  The README pages have no
 * counterpart: this is a deployment convenience of this library.
 *
 * Some callers may not call cudaMalloc or any other allocator: a plugin whose
 * host application owns the device-memory budget, or a latency-critical loop
 * where an allocation could synchronise the device and stall other streams.
 * They pass q, the caches, the tables and `out` as usual; the split-K
 * partials go to a scratch array compiled into the library instead of a
 * workspace.  Arguments and results are those of
 * photon_paged_attention_decode without `workspace` / `workspace_bytes`.
 *
 * Limits and behaviour:
 *   - the workspace the call would need,
 *     photon_paged_attention_workspace_size(num_seqs, num_q_heads, head_dim,
 *     max_context_len, partition_size), must not exceed
 *     PHOTON_STATIC_SCRATCH_BYTES; a larger request returns
 *     PHOTON_ERR_WORKSPACE and launches nothing;
 *   - allocates nothing: no cudaMalloc, cudaFree or allocating library call;
 *   - arguments are checked first, as photon_paged_attention_decode checks
 *     them (INVALID_ARG / UNSUPPORTED), then the size;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cached address belongs
 *     to the device's current context: a process that resets the device
 *     (cudaDeviceReset) must not call the library on it again;
 *   - every call on a device shares the one array, which keeps the previous
 *     call's partials; nothing in it needs to start at zero, but calls whose
 *     kernels overlap on the GPU (other streams, other threads) race on it and
 *     must be serialised by the caller.
 */
int photon_paged_attention_decode_static(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         float scale, void *out, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                         int32_t max_blocks_per_seq, int32_t max_context_len,
                                         int32_t partition_size, photon_dtype kv_dtype,
                                         photon_dtype out_dtype, photon_stream_t stream);

/*
 * photon_paged_attention_prefill -- causal attention of a chunk of new tokens
 * (a prompt, or a piece of one) over their sequences' pages: the other side
 * of the batched write for newly admitted requests.  Query token t belongs
 * to sequence token_seq[t] at position positions[t] and attends to that
 * sequence's tokens 0 .. positions[t] (their K/V must already be written):
 *   out[t][g][:] = sum_{j <= positions[t]} softmax_j(scale * <q[t][g][:], K[j]>) * V[j]
 * with the same GQA grouping, online softmax and split-K merge as the decode
 * call.  bf16 pools with head_dim 64 or 128 and G in {1, 2, 4, 8} run on the
 * tensor cores, query tokens grouped in row tiles of consecutive tokens of
 * one sequence that share every page they read (tokens of a sequence are
 * best kept contiguous and in position order; any order is correct).  Long
 * batches -- at least one 128-row tile (128/G tokens x G heads) per SM and
 * KV head -- run a tcgen05 kernel (accumulators in tensor memory) that
 * writes every row whole, with no split and no merge; shorter ones a kernel
 * of 16/G-token tiles that may use partitions coarser than partition_size
 * (a multiple of it, so the workspace below still suffices).  The result is
 * the same.  Other shapes handle each token as a decode query whose context
 * is its position + 1.
 *   q          device [num_tokens][num_q_heads][head_dim], kv_dtype, 16-B aligned
 *   token_seq  device int32 [num_tokens], rows of block_tables (0 .. num_seqs-1)
 *   positions  device int32 [num_tokens], each <= max_position
 *   out        device [num_tokens][num_q_heads][head_dim], out_dtype, 16-B aligned
 *   workspace  >= photon_paged_attention_workspace_size(num_tokens, num_q_heads,
 *              head_dim, max_position + 1, partition_size) bytes
 * Other arguments as photon_paged_attention_decode.  A token_seq entry out of
 * range yields a zero row and PHOTON_DEVERR_BLOCK_RANGE.
 */
int photon_paged_attention_prefill(const void *q, const int32_t *token_seq,
                                   const int32_t *positions, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables, float scale,
                                   void *out, int32_t num_tokens, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_blocks,
                                   int32_t max_blocks_per_seq, int32_t max_position,
                                   int32_t partition_size, photon_dtype kv_dtype,
                                   photon_dtype out_dtype, void *workspace,
                                   size_t workspace_bytes, photon_stream_t stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) KV cache with per-KV-head scales: half the bytes of bf16.
 *
 * Layout (one byte per value, E4M3 codes: 1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits, no infinities, largest finite 448):
 *   K pool [num_blocks][num_kv_heads][block_size][head_dim]   (as for bf16)
 *   V pool [num_blocks][num_kv_heads][head_dim][block_size]   (dims outer)
 * A stored code c of KV head h means decode(c) * k_scale[h] (K) or
 * decode(c) * v_scale[h] (V); scales are float32 device arrays [num_kv_heads].
 * ---------------------------------------------------------------------- */

/*
 * photon_kv_cache_write_fp8 -- the batched RoPE-fused write into FP8 pools:
 *   code = round_e4m3(RoPE(k[t][h]) / k_scale[h])   (K; fp64 rotation and quotient)
 *   code = round_e4m3(v[t][h] / v_scale[h])          (V)
 * round_e4m3 rounds to nearest, ties to even, and saturates at +-448.  V
 * codes are the nearest E4M3 of the exact quotient (exact midpoints to the
 * even code); K codes are that of the fp64 rotation's quotient.
 *   k, v      device [num_tokens][num_kv_heads][head_dim], in_dtype (f32 or bf16), 16-B aligned
 *   k_cache, v_cache  device FP8 pools (layout above), 16-B aligned
 * num_kv_heads <= 64 (PHOTON_ERR_UNSUPPORTED otherwise).  Other arguments and
 * errors as photon_kv_cache_write.
 */
int photon_kv_cache_write_fp8(const void *k, const void *v, const int32_t *positions,
                              const int64_t *slot_mapping, void *k_cache, void *v_cache,
                              const float *k_scale, const float *v_scale, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, photon_dtype in_dtype, float rope_theta,
                              photon_rope rope_style, photon_stream_t stream);

/*
 * photon_paged_attention_decode_fp8 -- photon_paged_attention_decode over FP8
 * pools: the same attention on the dequantised values.  q is bf16 (already
 * rotated); it is converted to f16 for the tensor cores, so |q| must stay
 * below 65504 (values below 2^-24 count as 0).  head_dim 64 or 128
 * (PHOTON_ERR_UNSUPPORTED otherwise); workspace as for the bf16 call.
 * When the context splits at all (workspace size > 0) the split-K pieces are
 * not fixed partitions but equal runs of pages, one per warp of the grid
 * (whatever the context lengths), at least partition_size tokens long except
 * where a sequence ends; the merge combines however many each row got.
 */
int photon_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, const int32_t *context_lens,
                                      float scale, void *out, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks,
                                      int32_t max_blocks_per_seq, int32_t max_context_len,
                                      int32_t partition_size, photon_dtype out_dtype,
                                      void *workspace, size_t workspace_bytes,
                                      photon_stream_t stream);

/*
 * photon_paged_attention_partial_fp8 -- the first half of
 * photon_paged_attention_decode_fp8, as photon_paged_attention_partial is of
 * photon_paged_attention_decode: writes `out` for single-partition sequences
 * and the split-K partials to the workspace; photon_paged_attention_reduce
 * (same out_dtype, workspace and partition_size) then merges them.  The pair,
 * called back to back on one stream with the same arguments, does exactly
 * what photon_paged_attention_decode_fp8 does.  Arguments and errors as
 * photon_paged_attention_decode_fp8.
 */
int photon_paged_attention_partial_fp8(const void *q, const void *k_cache, const void *v_cache,
                                       const float *k_scale, const float *v_scale,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       float scale, void *out, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int32_t max_blocks_per_seq, int32_t max_context_len,
                                       int32_t partition_size, photon_dtype out_dtype,
                                       void *workspace, size_t workspace_bytes,
                                       photon_stream_t stream);

/*
 * Reads (and, if clear != 0, resets) the sticky PHOTON_DEVERR_* bits of the
 * current device.  Synchronises the device: a diagnostic, not a hot-path call.
 * The bits only report: one left set does not change what later calls
 * compute.  The word's device address is looked up once per device and
 * cached, so after a device reset (cudaDeviceReset) the library must not be
 * called on that device again in the same process.
 */
int photon_device_errors(uint32_t *flags_out, int clear);

/*
 * Diagnostic of the failure path shared by every page pipeline: launches one
 * warp that waits, bounded by about budget_cycles SM clock cycles, on an
 * mbarrier phase that nothing completes.  The wait gives up, sets
 * PHOTON_DEVERR_WAIT_TIMEOUT (read it with photon_device_errors), lets any
 * copies in flight land and returns; the context stays usable.  Returns
 * PHOTON_ERR_INVALID_ARG for a zero budget, PHOTON_ERR_CUDA on a launch error.
 */
int photon_selftest_wait_timeout(uint32_t budget_cycles, photon_stream_t stream);

/* ------------------------------------------------------------------------
 * Ragged batch metadata (host side) -- what a two-phase scheduler step emits
 * ("Technical details > Continuous batching scheduler": running requests
 * continue, waiting requests are admitted; num_computed_tokens marks where
 * each request resumes).  All pointers here are HOST memory.
 * ---------------------------------------------------------------------- */

/* A pool of physical block ids 0..num_blocks-1 handed out from a free list
 * that starts in a seeded random order (splitmix64 + Fisher-Yates). */
typedef struct photon_block_pool photon_block_pool;

/* Creates a pool; *out receives the handle.  num_blocks in [1, 2^31-1]. */
int photon_block_pool_create(int64_t num_blocks, uint64_t seed, photon_block_pool **out);
void photon_block_pool_destroy(photon_block_pool *pool);
int64_t photon_block_pool_num_free(const photon_block_pool *pool);
/* Takes n blocks (all or none: PHOTON_ERR_POOL_EXHAUSTED leaves the pool as it was). */
int photon_block_pool_alloc(photon_block_pool *pool, int32_t n, int32_t *ids_out);
/* Returns n blocks; an id out of range or not currently allocated is rejected
 * (PHOTON_ERR_INVALID_ARG) and nothing is freed. */
int photon_block_pool_free(photon_block_pool *pool, const int32_t *ids, int32_t n);

/*
 * slot_mapping[t] = block_tables[token_seq[t]][positions[t] / bs] * bs + positions[t] % bs,
 * or -1 when the position is negative, past the row, or the entry is -1.
 *   block_tables  host int32 [num_seqs][max_blocks_per_seq]
 *   token_seq, positions  host int32 [num_tokens]
 *   slot_mapping  host int64 [num_tokens] (output)
 * A token_seq entry outside [0, num_seqs) is PHOTON_ERR_INVALID_ARG.
 */
int photon_slot_mapping(const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                        const int32_t *token_seq, const int32_t *positions, int32_t num_tokens,
                        int32_t block_size, int64_t *slot_mapping);

/*
 * Builds one step's metadata.  Sequence s has num_computed_tokens[s] tokens
 * in the cache and writes num_new_tokens[s] more this step (1 for a running
 * request's decode, the prompt length + 1 for a newly admitted one, 0 for an
 * idle row).  For each s, in order:
 *   - block_tables row s is grown from `pool` until it covers
 *     num_computed_tokens[s] + num_new_tokens[s] tokens (pool may be NULL if
 *     every row already covers its tokens);
 *   - the new tokens get positions num_computed_tokens[s] ..  + num_new - 1,
 *     token_seq = s, and their slot numbers;
 *   - context_lens[s] = num_computed_tokens[s] + num_new_tokens[s].
 *   block_tables  host int32 [num_seqs][max_blocks_per_seq], -1 = no block (in/out)
 *   token_seq, positions, slot_mapping  host outputs with room for max_tokens
 *   context_lens  host int32 [num_seqs] (output)
 *   *num_tokens_out, *max_context_len_out  totals (outputs)
 * Fails without partial effects on the pool if a row would overflow
 * max_blocks_per_seq (INVALID_ARG), tokens exceed max_tokens (INVALID_ARG)
 * or the pool runs out (POOL_EXHAUSTED).
 */
int photon_build_step_metadata(int32_t num_seqs, const int32_t *num_computed_tokens,
                               const int32_t *num_new_tokens, int32_t block_size,
                               int32_t *block_tables, int32_t max_blocks_per_seq,
                               photon_block_pool *pool, int32_t max_tokens, int32_t *token_seq,
                               int32_t *positions, int64_t *slot_mapping, int32_t *context_lens,
                               int32_t *num_tokens_out, int32_t *max_context_len_out);

/* ------------------------------------------------------------------------
 * Two-phase continuous-batching scheduler (host side).
 *
 * "Technical details > Continuous batching scheduler": phase 1 continues
 * every RUNNING request (no interruption), phase 2 admits WAITING requests
 * into the remaining capacity; requests move WAITING -> RUNNING -> FINISHED,
 * with PREEMPTED for requests that lost their blocks; num_computed_tokens
 * marks where a request resumes.
 *
 * A request knows L = prompt_len + generated tokens.  When scheduled it
 * processes tokens [num_computed_tokens, L) (all of them right after
 * admission, one per step afterwards) and holds ceil(L / block_size) blocks.
 * Phase 1 preempts the most recently admitted running request while the
 * pool cannot cover the running requests' next blocks: its blocks are freed,
 * num_computed_tokens drops to 0 and it goes back to the FRONT of the waiting
 * queue.  Phase 2 admits waiting requests first come first served while a
 * batch slot, the step's token budget and enough free blocks remain; the
 * first request that does not fit ends the phase.
 * ---------------------------------------------------------------------- */
typedef struct photon_scheduler photon_scheduler;

typedef enum {
  PHOTON_REQ_WAITING = 0,
  PHOTON_REQ_RUNNING = 1,
  PHOTON_REQ_FINISHED = 2,
  PHOTON_REQ_PREEMPTED = 3 /* waiting again, to recompute from token 0 */
} photon_request_state;

typedef struct {
  int32_t max_running;        /* batch slots: running requests per step */
  int32_t max_step_tokens;    /* token budget of a step (admissions stop at it) */
  int32_t max_blocks_per_seq; /* width of a block-table row */
  int32_t block_size;         /* tokens per block (16 for the kernels) */
} photon_scheduler_config;

/* One step's batch, written into caller-owned HOST arrays.  Capacities:
 * max_seqs >= config.max_running, max_tokens >= config.max_step_tokens.
 * Row i of the batch is the i-th running request in admission order.
 * block_tables is updated incrementally when the same buffer is passed again:
 * a row that holds the same request as in the previous batch only receives
 * its newly allocated blocks, so the caller must not modify the buffer between
 * steps (passing a different buffer makes the next batch write every row). */
typedef struct {
  int32_t max_seqs;
  int32_t max_tokens;
  int64_t *request_ids;    /* [max_seqs] */
  int32_t *num_new_tokens; /* [max_seqs] tokens processed this step */
  int32_t *context_lens;   /* [max_seqs] L after this step's tokens */
  int32_t *block_tables;   /* [max_seqs][max_blocks_per_seq], -1 padded */
  int32_t *token_seq;      /* [max_tokens] batch row of each processed token */
  int32_t *positions;      /* [max_tokens] its position */
  int64_t *slot_mapping;   /* [max_tokens] its cache slot */
  int32_t num_seqs;        /* outputs */
  int32_t num_tokens;
  int32_t max_context_len;
  int32_t num_preempted;
  int32_t num_admitted;
} photon_step_batch;

/* Creates a scheduler drawing blocks from `pool` (which must outlive it). */
int photon_scheduler_create(const photon_scheduler_config *config, photon_block_pool *pool,
                            photon_scheduler **out);
/* Destroys the scheduler; blocks its requests still hold go back to the pool. */
void photon_scheduler_destroy(photon_scheduler *sched);
/* Queues a request (WAITING).  Rejected (INVALID_ARG) if the id is in use,
 * a length is not positive, prompt_len + max_new_tokens needs more than
 * max_blocks_per_seq blocks, or its longest recompute (prompt_len +
 * max_new_tokens - 1 tokens) exceeds max_step_tokens; POOL_EXHAUSTED if it
 * needs more blocks than the pool holds. */
int photon_scheduler_add_request(photon_scheduler *sched, int64_t request_id, int32_t prompt_len,
                                 int32_t max_new_tokens);
/* Plans one step (both phases) and fills `batch`.  Fails (INVALID_ARG) while
 * the previous step has not been completed. */
int photon_scheduler_schedule(photon_scheduler *sched, photon_step_batch *batch);
/* Marks the planned step done: every scheduled request has computed its
 * tokens and generated one more; requests reaching max_new_tokens finish and
 * free their blocks. */
int photon_scheduler_complete_step(photon_scheduler *sched);
/* State, num_computed_tokens and generated-token count of a request. */
int photon_scheduler_request_state(const photon_scheduler *sched, int64_t request_id,
                                   int32_t *state, int32_t *num_computed_tokens,
                                   int32_t *num_generated);
/* Queue sizes. */
int photon_scheduler_counts(const photon_scheduler *sched, int32_t *num_waiting,
                            int32_t *num_running, int32_t *num_finished);

#ifdef __cplusplus
}
#endif

#endif /* PHOTON_H */
