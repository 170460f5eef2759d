// Tensor-core split-K paged decode attention for bf16 KV (head_dim 64, 128).
//
// Same computation and the same partial/merge contract as the CUDA-core
// kernel in paged_decode.cuh (PhotonInfer README, "Key features >
// GPU-optimised kernels": batched paged attention with a numerically stable
// softmax), organised for sm_103a:
//
//  * Every warp is an independent worker: it owns whole work items (sequence
//    x KV head x context partition) and its own ring of ST shared-memory
//    stages.  Global warp w of W takes item w first, then, with a workspace,
//    the next unclaimed item from a counter in the workspace (see DecodeCtl:
//    warps that run faster take more items), else items w + W, w + 2W, ....
//    There is no CTA-wide barrier after set-up.  Lane 0 walks the warp's
//    stream of pages ST pages ahead of the compute, across item boundaries,
//    so the copy pipeline never drains between items.
//  * On long steps the producer also prefetches the pages l2_lookahead ahead
//    of its ring into L2 (a bulk prefetch on the TMA engine, issued after the
//    demand copy), which puts more bytes in flight per SM than the ring,
//    bounded by shared memory, can hold.
//  * A page's K rows and V rows each arrive by one TMA tensor copy
//    (cp.async.bulk.tensor) from a 2-D/3-D view of the pool,
//    [num_blocks*H_kv*bs rows] x [d], with the 128-byte swizzle: fragment
//    loads from shared memory below are then free of bank conflicts.
//  * S^T = Q K^T on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//    accumulate): the G query heads of the group are the 16-row M side
//    (rows G..15 are zero), 16 tokens of a page are N, head_dim is K.  The
//    head dimensions are visited in a per-thread permuted order (the same for
//    q and K, so dot products are unchanged) so each thread reads whole
//    16-byte chunks.
//  * Online softmax in base 2 on the accumulator fragments (page max by two
//    shuffles among the four lanes of a row), then O += P V on the tensor
//    cores with P taken straight from the score fragments (no shuffles).  P
//    is split into a bf16 high part and a bf16 remainder, two MMAs, so the
//    probabilities keep ~16 significant bits instead of 8.  V fragments are
//    assembled with byte permutes from 16-byte loads.
//  * At the end of an item the warp writes the normalised output (single
//    partition) or the unnormalised partial with its running max and sum.
#pragma once

#include <atomic>
#include <cuda.h>

#include <climits>

#include "common.cuh"
#include "internal.h"
#include "paged_decode.cuh"

namespace photon {

template <int D, int G, int NW, int ST>
struct MmaCfg {
  static_assert(D == 64 || D == 128, "tensor-core path: head_dim 64 or 128");
  static_assert(G >= 1 && G <= 8, "tensor-core path: at most 8 query heads per KV head");
  static constexpr int PAGE_BYTES = kBlockSize * D * 2;  // K (or V) rows of one page
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int KT = D / 16;      // k-steps of Q K^T
  static constexpr int KW = D / 8;       // 32-bit words of a K row per thread (2 per k-step)
  static constexpr int KCH = KW / 4;     // 16-byte chunks of a K row per thread
  static constexpr int MT = D / 16;      // m-tiles (16 head dims each) of V^T P^T
  static constexpr int HALVES = D / 64;  // V page halves of 64 dims (TMA box layout)
  static constexpr int SMEM = NW * ST * STAGE_BYTES + NW * ST * 8 + 1024;  // +1 KiB for alignment
  // CTAs per SM that shared memory allows (227 KiB per SM, 2 KiB static and
  // reserved per CTA); handed to the compiler as the register target at d 64,
  // where without it ptxas spilled
  static constexpr int MIN_CTAS = (227 * 1024) / (SMEM + 2048);
};

__device__ __forceinline__ uint32_t swz128(uint32_t off) {
  // 128-byte swizzle of the TMA engine: the 16-byte chunk index (bits 4-6)
  // is XORed with the 128-byte line index within a 1 KiB atom (bits 7-9).
  return off ^ (((off >> 7) & 7u) << 4);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                               uint32_t b1) {
  // rows 8..15 of A are zero (a1 = a3 = 0)
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void tma_load_page(void *dst, const CUtensorMap *map, int rank3, int row,
                                              uint64_t *bar, uint64_t policy);

__device__ __forceinline__ void mma_bf16_16816_full(float (&d)[4], uint32_t a0, uint32_t a1,
                                                    uint32_t a2, uint32_t a3, uint32_t b0,
                                                    uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// K page: rows of D values in order (D = 64: 2-D box {64, 16};
// D = 128: 3-D box {64, 2, 16}, i.e. [16 rows][2 x 64]).
template <int D>
__device__ __forceinline__ void tma_load_k_page(void *dst, const CUtensorMap *map, int row,
                                                uint64_t *bar, uint64_t policy) {
  tma_load_page(dst, map, D > 64, row, bar, policy);
}

// V page: D/64 halves of [16 rows][64 values] in shared memory, each half
// one 2-D copy (box {64, 16}) of a {D, rows} view at x = 0, 64, ...
template <int D>
__device__ __forceinline__ void tma_load_v_page(void *dst, const CUtensorMap *map, int row,
                                                uint64_t *bar, uint64_t policy) {
#pragma unroll
  for (int hh = 0; hh < D / 64; ++hh)
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(
            static_cast<unsigned char *>(dst) + hh * kBlockSize * 128)),
        "l"(map), "r"(64 * hh), "r"(row), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_page(void *dst, const CUtensorMap *map, int rank3, int row,
                                              uint64_t *bar, uint64_t policy) {
  if (rank3)
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(0), "r"(0), "r"(row), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(0), "r"(row), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Position of one warp in its stream of (item, page).  An item is one
// sequence x KV head x piece of its context: pages pg0 .. pg0 + n_pages - 1,
// piece p of the P_s pieces of that (sequence, KV head).
struct Walker {
  int item;            // global item index (fixed partitions)
  int cur_s, cur_base; // sequence cursor: first partition index of sequence cur_s
  int s, p, h, ctx, P_s, tok0, tok1, pg0, n_pages;
  int page;            // next page of the item
  bool valid;
  // page-balanced pieces: the warp's run [u, u_end) of the unit stream (q
  // units per group), the current sequence's first unit seq_base.  The
  // stream has at most INT32_MAX / 2 units.
  int u, u_end, q, seq_base;
};

// Token and page range of partition w.p of sequence w.s (context w.ctx).
__device__ __forceinline__ void item_fields(Walker &w, const DecodeArgs &a) {
  w.P_s = w.ctx <= 0 ? 1 : (w.ctx + a.partition_size - 1) / a.partition_size;
  w.tok0 = w.p * a.partition_size;
  w.tok1 = min(w.tok0 + a.partition_size, w.ctx);
  w.pg0 = w.tok0 / kBlockSize;
  w.n_pages = w.tok1 > w.tok0 ? (w.tok1 - w.tok0 + kBlockSize - 1) / kBlockSize : 0;
  w.page = 0;
}

// Decode batches of up to this many sequences have their context lengths
// staged in shared memory (1 KiB).
constexpr int kCtxStage = 256;
__device__ __forceinline__ bool ctx_staged(const DecodeArgs &a) {
  return a.query_positions == nullptr && a.num_seqs <= kCtxStage;
}

// Finds (sequence, partition) of w.item with a warp-wide scan over
// context_lens starting at the cursor; sets w.valid = false past the end.
// staged: a copy of a decode batch's context_lens (in shared memory), used
// when ctx_staged(a); NULL: always read them (or the prefill positions) from a.
__device__ __forceinline__ void walker_locate(Walker &w, const DecodeArgs &a, int lane,
                                              unsigned int *err, const int32_t *staged = nullptr) {
  const int pw = w.item / a.num_kv_heads;
  w.h = w.item - pw * a.num_kv_heads;
  w.valid = false;
  while (w.cur_s < a.num_seqs) {
    const int s = w.cur_s + lane;
    int P = 0, c = 0;
    if (s < a.num_seqs) {
      c = (staged && ctx_staged(a)) ? staged[s] : seq_context(a, s, err);
      if (c > a.ctx_cap) {
        atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
        c = a.ctx_cap;
      }
      c = c < 0 ? 0 : c;
      P = c <= 0 ? 1 : (c + a.partition_size - 1) / a.partition_size;
    }
    int incl = P;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, s < a.num_seqs && w.cur_base + incl > pw);
    if (hit) {
      const int L = __ffs(hit) - 1;
      w.cur_base += __shfl_sync(0xffffffffu, incl - P, L);
      w.ctx = __shfl_sync(0xffffffffu, c, L);
      w.cur_s += L;
      w.valid = true;
      break;
    }
    w.cur_base += __shfl_sync(0xffffffffu, incl, 31);
    w.cur_s += 32;
  }
  if (!w.valid) return;
  w.s = w.cur_s;
  w.p = pw - w.cur_base;
  item_fields(w, a);
}

// ---- page-balanced pieces (decode with a workspace) ----------------------
// The unit stream lists, sequence by sequence, one unit per page of the
// context (an empty context still one unit, whose piece writes the zero
// row).  With U units and WG groups of H_kv consecutive warps, group j takes
// the run [j q, (j + 1) q), q = max(ceil(U / WG), partition_size / 16), and
// its warp h works on KV head h.  Every warp gets the same number of pages
// whatever the context lengths; the H_kv warps of a group read the same
// blocks at about the same time (a block's heads are contiguous in the
// pool); a sequence of u units meets at most ceil(u / q) + 1 <=
// max_partitions runs.  The piece of the run starting at unit u in the
// sequence starting at unit A is piece floor(u / q) - floor(A / q) of
// floor((A + u_s - 1) / q) - floor(A / q) + 1.  A run's pieces are
// consecutive sequences, so after the first (located by a scan of the
// context lengths) the walker steps to the next sequence.

__device__ __forceinline__ int units_of(int ctx) {
  return ctx <= 0 ? 1 : (ctx + kBlockSize - 1) / kBlockSize;
}

__device__ __forceinline__ int balanced_ctx(const DecodeArgs &a, int s, unsigned int *err) {
  int c = a.context_lens[s];
  if (c > a.ctx_cap) {
    atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
    c = a.ctx_cap;
  }
  return c < 0 ? 0 : c;
}

// Item fields of the piece starting at unit w.u of sequence w.s (context
// w.ctx, first unit w.seq_base).
__device__ __forceinline__ void balanced_fill(Walker &w) {
  const int us = units_of(w.ctx);
  const int pb = w.u - w.seq_base;
  const int end = min(w.seq_base + us, w.u_end);
  const int n_s = w.ctx > 0 ? us : 0;  // real pages
  w.pg0 = pb;
  w.n_pages = max(0, min(n_s, pb + (end - w.u)) - pb);
  const int first = w.seq_base / w.q;
  w.p = w.u / w.q - first;
  w.P_s = (w.seq_base + us - 1) / w.q - first + 1;
  w.tok0 = pb * kBlockSize;
  w.tok1 = w.ctx;
  w.page = 0;
}

// At the start of a balanced launch the grid's threads prefetch the block
// tables into L2, one 128-byte line each (tables up to 8 MiB): a warp's
// first block-table load then follows its context-length scan from L2
// rather than DRAM.
__device__ __forceinline__ void prefetch_tables_l2(const DecodeArgs &a) {
  const int64_t lines = (static_cast<int64_t>(a.num_seqs) * a.max_blocks_per_seq * 4 + 127) / 128;
  if (lines > (int64_t{1} << 16)) return;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t l = i; l < lines; l += static_cast<int64_t>(gridDim.x) * blockDim.x)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(a.block_tables) + l * 128)
                 : "memory");
}

// First piece of global warp gw of W.
__device__ __forceinline__ void balanced_start(Walker &w, const DecodeArgs &a, int lane,
                                               unsigned int *err, int gw, int W) {
  int tot = 0;
  for (int s0 = lane; s0 < a.num_seqs; s0 += 128) {  // four independent loads per round
    int c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = s0 + 32 * k < a.num_seqs ? a.context_lens[s0 + 32 * k] : INT_MIN;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (c[k] != INT_MIN) {
        if (c[k] > a.ctx_cap) {
          atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
          c[k] = a.ctx_cap;
        }
        tot += units_of(c[k]);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const int groups = W / a.num_kv_heads;
  const int j = gw / a.num_kv_heads;
  w.h = gw - j * a.num_kv_heads;
  w.valid = j < groups;
  if (!w.valid) return;
  w.q = max((tot + groups - 1) / groups, max(a.partition_size / kBlockSize, 1));
  const int64_t u0 = static_cast<int64_t>(j) * w.q;  // may pass the stream's end
  w.valid = u0 < tot;
  if (!w.valid) return;
  w.u = static_cast<int>(u0);
  w.u_end = static_cast<int>(min(u0 + w.q, static_cast<int64_t>(tot)));
  // the sequence holding unit u: forward scan, 32 sequences per step (bounded
  // by the batch: lengths changed under the kernel end the run instead)
  int base = 0;
  w.valid = false;
  for (int s0 = 0; s0 < a.num_seqs; s0 += 32) {
    const int s = s0 + lane;
    const int c = s < a.num_seqs ? balanced_ctx(a, s, err) : 0;
    const int un = s < a.num_seqs ? units_of(c) : 0;
    int incl = un;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, s < a.num_seqs && base + incl > w.u);
    if (hit) {
      const int L = __ffs(hit) - 1;
      w.s = s0 + L;
      w.seq_base = base + __shfl_sync(0xffffffffu, incl - un, L);
      w.ctx = __shfl_sync(0xffffffffu, c, L);
      w.valid = true;
      break;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (w.valid) balanced_fill(w);
}

// Next piece of the warp's run (the next sequence), or valid = false at its end.
__device__ __forceinline__ void balanced_next(Walker &w, const DecodeArgs &a, unsigned int *err) {
  w.seq_base += units_of(w.ctx);
  w.u = w.seq_base;
  w.valid = w.u < w.u_end;
  if (!w.valid) return;
  if (++w.s >= a.num_seqs) {  // only if the lengths changed under the kernel
    w.valid = false;
    return;
  }
  w.ctx = balanced_ctx(a, w.s, err);
  balanced_fill(w);
}

// BAL: page-balanced pieces (kernels instantiated per mode, so that each
// keeps only its own walker state in registers).
template <bool BAL>
__device__ __forceinline__ void walker_start(Walker &w, const DecodeArgs &a, int lane,
                                             unsigned int *err, int gw, int W) {
  if constexpr (BAL) {
    balanced_start(w, a, lane, err, gw, W);
  } else {
    w.item = gw;
    w.cur_s = w.cur_base = 0;
    walker_locate(w, a, lane, err);
  }
}

template <bool BAL>
__device__ __forceinline__ void walker_next(Walker &w, const DecodeArgs &a, int lane,
                                            unsigned int *err, int W) {
  if constexpr (BAL) {
    balanced_next(w, a, err);
  } else {
    w.item += W;
    walker_locate(w, a, lane, err);
  }
}

// ---- dynamic item order (decode with a workspace) -------------------------
// After its first item (its own index) a warp claims the next unclaimed item
// from the workspace's control block (DecodeCtl), so the warps that the memory
// system serves faster take more items and the grid runs out of work all at
// once rather than at the ends of fixed shares.

// The launch's first thread: both counters tagged, at zero.
__device__ __forceinline__ void ctl_publish(DecodeCtl *ctl) {
  *reinterpret_cast<volatile unsigned long long *>(&ctl->next) = kCtlTag;
  *reinterpret_cast<volatile unsigned long long *>(&ctl->done) = kCtlTag;
}

__device__ __forceinline__ bool ctl_tagged(unsigned long long w) {
  return (w >> kCtlCountBits) == (kCtlTag >> kCtlCountBits);
}

// Count taken from a counter: `first` is the word a first atomic add returned
// (its round trip hidden by the caller); adds that came before the
// launch's ctl_publish are repeated (bounded).  -1 if that gave up.
__device__ __forceinline__ int ctl_take(unsigned long long *counter, unsigned long long first,
                                        unsigned int *err) {
  if (ctl_tagged(first)) return static_cast<int>(first & ((1ull << kCtlCountBits) - 1));
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(256);
    const unsigned long long w = atomicAdd(counter, 1ull);
    if (ctl_tagged(w)) return static_cast<int>(w & ((1ull << kCtlCountBits) - 1));
    if (clock64() - t0 > kWaitBudgetCycles) {
      atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
      return -1;
    }
  }
}

// At the warp's exit, with the word its add to `done` returned: the last of
// the grid's `warps` to leave returns both counters to 0.
__device__ __forceinline__ void ctl_close(DecodeCtl *ctl, unsigned long long ticket, int warps,
                                          unsigned int *err) {
  if (ctl_take(&ctl->done, ticket, err) == warps - 1) {
    ctl->next = 0ull;
    ctl->done = 0ull;
  }
}

// DYN: dynamic item order through a.ctl (else every total_warps-th item).
// Launch bounds: at d 64 the shared-memory occupancy as the register target
// (MIN_CTAS); at d 128 none (0), where the compiler's own choice fits (with
// the target, 168 registers and spills: Qwen3 batch-64 kernel 92.8 -> 95.9 us).
template <int D, int G, int NW, int ST, bool DYN>
__global__ void __launch_bounds__(NW * 32, D == 64 ? MmaCfg<D, G, NW, ST>::MIN_CTAS : 0)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a,
                            unsigned int *err) {
  using C = MmaCfg<D, G, NW, ST>;
  extern __shared__ unsigned char smem_raw[];
  // 1 KiB alignment: the 128-byte swizzle pattern repeats every 1 KiB
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair
  unsigned char *stages = smem + warp * ST * C::STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * ST * C::STAGE_BYTES) + warp * ST;
  const uint32_t stages_s = smem_addr(stages);

  if (lane == 0) {
    for (int i = 0; i < ST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
  }
  __syncwarp();
  pdl_launch_dependents();

  const uint64_t policy = l2_evict_first_policy();
  const uint64_t keep_policy = l2_evict_last_policy();
  const int total_warps = gridDim.x * NW;
  const int first_item = blockIdx.x * NW + warp;

  // Per-thread byte offsets of its fragment chunks inside a stage (swizzled).
  // K page: rows of D values.  Thread (g, c) reads rows g and 8+g, chunks
  // KCH*c .. KCH*c + KCH - 1 (head dims in the permuted order of the q
  // fragments).
  uint32_t koff[2][C::KCH];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < C::KCH; ++i)
      koff[nt][i] = swz128((8 * nt + g) * C::ROW_BYTES + (C::KCH * c + i) * 16);
  // V page: D/64 halves of [16 rows][64 values] (each row 128 bytes).  Thread
  // (g, c) reads tokens 2c, 2c+1, 2c+8, 2c+9, chunk g of every half.
  uint32_t voff[4][C::HALVES];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int hh = 0; hh < C::HALVES; ++hh) {
      const int row = 2 * c + (r & 1) + 8 * (r >> 1);
      voff[r][hh] = C::PAGE_BYTES + hh * (kBlockSize * 128) + swz128(row * 128 + g * 16);
    }

  // Fixed order (single-wave grids, whose warps have about one item each and
  // are bound by start-up): a decode batch's context lengths are read once
  // per CTA into shared memory for the warps' scans (single-request step
  // 4.64 -> 4.3 us per layer; no change on full grids, which skip it).
  __shared__ int32_t ctx_s[DYN ? 1 : kCtxStage];
  if (!DYN && ctx_staged(a)) {
    for (int i = threadIdx.x; i < a.num_seqs; i += NW * 32) ctx_s[i] = a.context_lens[i];
    __syncthreads();
  }
  // The producer walks the warp's items (first its own index, then the next
  // unclaimed one (DYN) or every total_warps-th) and records each, and the
  // end, in a ring of records spread over the lanes (lane j: records j mod
  // 32); the consumer, a few pages behind, replays them.
  Walker prod, cons;
  prod.item = first_item;
  prod.cur_s = prod.cur_base = 0;
  walker_locate(prod, a, lane, err, DYN ? nullptr : ctx_s);
  int rec_s = -1, rec_h = 0, rec_p = 0, rec_ctx = 0;  // this lane's record (s -1: the end)
  uint32_t n_rec = 0, n_cons_item = 0;  // records written; the consumer's current item
  auto record = [&]() {
    if (lane == static_cast<int>(n_rec % 32)) {
      rec_s = prod.valid ? prod.s : -1;
      rec_h = prod.h;
      rec_p = prod.p;
      rec_ctx = prod.ctx;
    }
    ++n_rec;
  };
  record();
  // Everything above reads only the batch's metadata (context lengths, block
  // tables), which no kernel of the step writes: under programmatic launch it
  // runs beside the preceding kernel.  The first item's block-table entries go
  // to L2 meanwhile.  Pages, the query and the workspace wait for it.
  if (lane < 2 && prod.valid && prod.n_pages > 0 && prod.pg0 + 32 * lane < a.max_blocks_per_seq)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.block_tables +
                                                 seq_table_row(a, prod.s) * a.max_blocks_per_seq +
                                                 prod.pg0 + 32 * lane)
                 : "memory");
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (a.seg_count) a.seg_count[static_cast<int64_t>(a.num_seqs) * a.num_q_heads] = 0;  // the merge's mode
    if constexpr (DYN) ctl_publish(a.ctl);
  }
  // DYN: lane 0's claim in flight (items past the first ones), made one item
  // ahead so that the counter's round trip hides behind the current item;
  // lane 0's add to the count of warps that left, made when the claims run out
  unsigned long long claim = 0, ticket = 0;
  bool have_claim = false, left = false;
  auto claim_next = [&]() {
    if (lane == 0) claim = atomicAdd(&a.ctl->next, 1ull);
    have_claim = true;
  };
  auto leave = [&]() {
    if (lane == 0) ticket = atomicAdd(&a.ctl->done, 1ull);
    left = true;
  };
  uint32_t n_issued = 0, n_consumed = 0, valid_bits = 0;
  // block-table window of the producer's item: lane j holds the entry of page
  // bt_base + j (loaded once per 32 pages instead of once per page)
  int bt_base = INT_MIN / 2, bt_reg = -1;
  int pf_next = 0;  // next page of the producer's item to prefetch into L2

  // Moves the producer past items whose pages are all issued, recording each
  // new item (and the end); false when it has no page to issue now (the end,
  // or 32 records ahead of the consumer).
  auto prod_advance = [&]() -> bool {
    while (prod.valid && prod.page >= prod.n_pages) {
      if (n_rec - n_cons_item >= 32) return false;
      if constexpr (DYN) {
        if (!have_claim) claim_next();
        int idx = 0;
        if (lane == 0) {
          idx = ctl_take(&a.ctl->next, claim, err);
          idx = idx < 0 ? INT_MAX / 2 : idx;  // gave up: no more items
        }
        prod.item = total_warps + __shfl_sync(0xffffffffu, idx, 0);
      } else {
        prod.item += total_warps;
      }
      walker_locate(prod, a, lane, err, DYN ? nullptr : ctx_s);
      if constexpr (DYN) {
        if (prod.valid) {
          claim_next();
        } else {  // no more claims: the warp leaves the count now
          leave();
        }
      }
      // the item's query rows go to L2 now, a few pages before the consumer loads them
      if (lane == 0 && prod.valid && prod.n_pages > 0)
        bulk_prefetch_l2(static_cast<const __nv_bfloat16 *>(a.q) +
                             (static_cast<int64_t>(prod.s) * a.num_q_heads + prod.h * G) * D,
                         G * D * 2);
      record();
      bt_base = INT_MIN / 2;
    }
    return prod.valid;
  };

  // Issues the producer's next page (skipping items without pages).  Lane 0
  // copies; every lane keeps the walker.  Returns false when none is left
  // for now.
  auto issue_next = [&]() -> bool {
    if (!prod_advance()) return false;
    // pages [pf_next, pf_end) of the item go to L2 now: at the item's first
    // page the whole lookahead, then one page per issued page
    if (prod.page == 0) pf_next = 1;
    const int pf_end = a.l2_lookahead > 0 ? min(prod.page + a.l2_lookahead + 1, prod.n_pages) : 0;
    if (prod.page - bt_base >= 32 || pf_end - 1 - bt_base >= 32) {
      bt_base = prod.page;
      bt_reg = bt_base + lane < prod.n_pages
                   ? a.block_tables[seq_table_row(a, prod.s) * a.max_blocks_per_seq +
                                    prod.pg0 + bt_base + lane]
                   : -1;
    }
    const int blk = __shfl_sync(0xffffffffu, bt_reg, prod.page - bt_base);
    const uint32_t st = n_issued % ST;
    if (lane == 0) {
      if (blk >= 0 && blk < a.num_blocks) {
        const int row = (blk * a.num_kv_heads + prod.h) * kBlockSize;
        unsigned char *dst = stages + st * C::STAGE_BYTES;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES);
        tma_load_k_page<D>(dst, &tm_k, row, &bars[st], policy);
        tma_load_v_page<D>(dst + C::PAGE_BYTES, &tm_v, row, &bars[st], policy);
        valid_bits |= 1u << st;
      } else {
        atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
        mbar_arrive(&bars[st]);
        valid_bits &= ~(1u << st);
      }
    }
    // after the demand copy, so that it never queues behind a prefetch
    for (; pf_next < pf_end; ++pf_next) {
      const int pb = __shfl_sync(0xffffffffu, bt_reg, pf_next - bt_base);
      if (lane == 0 && pb >= 0 && pb < a.num_blocks) {
        const int64_t off = (static_cast<int64_t>(pb) * a.num_kv_heads + prod.h) * C::PAGE_BYTES;
        bulk_prefetch_l2(static_cast<const unsigned char *>(a.k_cache) + off, C::PAGE_BYTES);
        bulk_prefetch_l2(static_cast<const unsigned char *>(a.v_cache) + off, C::PAGE_BYTES);
      }
    }
    ++prod.page;
    ++n_issued;
    return true;
  };

  for (int k = 0; k < ST; ++k)
    if (!issue_next()) break;
  if constexpr (DYN)
    if (!prod.valid && !left) leave();  // nothing at all for this warp

  // the consumer's item from its record
  auto cons_enter = [&]() {
    const int src = static_cast<int>(n_cons_item % 32);
    cons.s = __shfl_sync(0xffffffffu, rec_s, src);
    cons.h = __shfl_sync(0xffffffffu, rec_h, src);
    cons.p = __shfl_sync(0xffffffffu, rec_p, src);
    cons.ctx = __shfl_sync(0xffffffffu, rec_ctx, src);
    cons.valid = cons.s >= 0;
    if (cons.valid) item_fields(cons, a);
  };
  cons_enter();

  // accumulators of the current item
  uint32_t qa[C::KT][2];   // A fragments of q (row g < G), words KW*c + 2kt (+1)
  float o[C::MT][4];       // O^T fragments: (dim, heads 2c and 2c+1), see the store below
  float m_run = -INFINITY, l_run = 0.f;  // of head g, over this lane's tokens

  while (cons.valid) {
    if (cons.page == 0) {
      // new item: load the query group (bf16 words, permuted head dims)
      uint32_t qw[C::KW];
      if (g < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const __nv_bfloat16 *>(a.q) +
            (static_cast<int64_t>(cons.s) * a.num_q_heads + cons.h * G + g) * D + C::KW * 2 * c);
#pragma unroll
        for (int i = 0; i < C::KCH; ++i) {
          const uint4 v = src[i];
          qw[4 * i] = v.x;
          qw[4 * i + 1] = v.y;
          qw[4 * i + 2] = v.z;
          qw[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < C::KW; ++i) qw[i] = 0u;
      }
#pragma unroll
      for (int kt = 0; kt < C::KT; ++kt) {
        qa[kt][0] = qw[2 * kt];
        qa[kt][1] = qw[2 * kt + 1];
      }
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    if (cons.page < cons.n_pages) {
      const uint32_t st = n_consumed % ST;
      const uint32_t par = (n_consumed / ST) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], par, kWaitBudgetCycles));
      if (!ok) {
        if (lane == 0) atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
        drain_async_copies();
        break;
      }
      const bool valid = __shfl_sync(0xffffffffu, (valid_bits >> st) & 1u, 0) != 0;
      const int page_tok0 = (cons.pg0 + cons.page) * kBlockSize;
      const int nvalid = valid ? min(kBlockSize, cons.tok1 - page_tok0) : 0;
      if (nvalid > 0) {
        const uint32_t base = stages_s + st * C::STAGE_BYTES;
        // ---- S^T = Q K^T (M = query heads, N = tokens in two n-tiles of 8)
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t kw[C::KW];
#pragma unroll
          for (int i = 0; i < C::KCH; ++i)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(kw[4 * i]), "=r"(kw[4 * i + 1]), "=r"(kw[4 * i + 2]),
                           "=r"(kw[4 * i + 3])
                         : "r"(base + koff[nt][i]));
          s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
          for (int kt = 0; kt < C::KT; ++kt)
            mma_bf16_16816(s[nt], qa[kt][0], qa[kt][1], kw[2 * kt], kw[2 * kt + 1]);
        }
        // ---- online softmax for head g over tokens 8nt + 2c + j
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float v = s[nt][j] * a.scale_log2;
            if (8 * nt + 2 * c + j >= nvalid) v = -INFINITY;
            s[nt][j] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = exp2f(m_run - m_new);
        m_run = m_new;
        float ps = 0.f;
        uint32_t ph[2], pl[2];  // P^T B fragments: (tokens 2c, 2c+1) of n-tile nt, head g
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float p0 = exp2f(s[nt][0] - m_new);
          const float p1 = exp2f(s[nt][1] - m_new);
          ps += p0 + p1;
          ph[nt] = pack_bf16(p0, p1);
          pl[nt] = pack_bf16(p0 - bf16_lo(ph[nt]), p1 - bf16_hi(ph[nt]));
        }
        l_run = fmaf(l_run, alpha, ps);
        // the O^T columns this lane holds are heads 2c and 2c+1
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * c);
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          o[mt][0] *= a0;
          o[mt][1] *= a1;
          o[mt][2] *= a0;
          o[mt][3] *= a1;
        }
        // ---- O^T += V^T P^T (M = head dims, N = query heads, K = 16 tokens)
        uint32_t vw[4][4 * C::HALVES];  // tokens 2c, 2c+1, 2c+8, 2c+9: dims 8g.. of each half
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(vw[r][4 * hh]), "=r"(vw[r][4 * hh + 1]), "=r"(vw[r][4 * hh + 2]),
                           "=r"(vw[r][4 * hh + 3])
                         : "r"(base + voff[r][hh]));
        if (nvalid < kBlockSize) {  // rows past the context may hold any bits
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = 2 * c + (r & 1) + 8 * (r >> 1);
            if (row >= nvalid)
#pragma unroll
              for (int i = 0; i < 4 * C::HALVES; ++i) vw[r][i] = 0u;
          }
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          uint32_t a_0, a_1, a_2, a_3;
          if (C::HALVES == 1) {
            // m-tile mt: rows g -> dim 8g + 2mt, g+8 -> dim 8g + 2mt + 1 (word mt)
            a_0 = __byte_perm(vw[0][mt], vw[1][mt], 0x5410u);
            a_1 = __byte_perm(vw[0][mt], vw[1][mt], 0x7632u);
            a_2 = __byte_perm(vw[2][mt], vw[3][mt], 0x5410u);
            a_3 = __byte_perm(vw[2][mt], vw[3][mt], 0x7632u);
          } else {
            // m-tile mt: rows g -> dim 8g + mt (half 0), g+8 -> dim 64 + 8g + mt (half 1)
            const int ww = mt >> 1;
            const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
            a_0 = __byte_perm(vw[0][ww], vw[1][ww], sel);
            a_1 = __byte_perm(vw[0][4 + ww], vw[1][4 + ww], sel);
            a_2 = __byte_perm(vw[2][ww], vw[3][ww], sel);
            a_3 = __byte_perm(vw[2][4 + ww], vw[3][4 + ww], sel);
          }
          mma_bf16_16816_full(o[mt], a_0, a_1, a_2, a_3, ph[0], ph[1]);
          mma_bf16_16816_full(o[mt], a_0, a_1, a_2, a_3, pl[0], pl[1]);
        }
      }
      __syncwarp();
      ++n_consumed;
      ++cons.page;
      issue_next();
      if constexpr (DYN)  // the first claim, once the warp's first page is in
        if (!have_claim && prod.valid) claim_next();
    }

    if (cons.page >= cons.n_pages) {
      // ---- item done: totals of head g, moved to the lanes holding heads 2c, 2c+1
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const float l0 = __shfl_sync(0xffffffffu, l, 8 * c);
      const float l1 = __shfl_sync(0xffffffffu, l, 8 * c + 4);
      const float m0 = __shfl_sync(0xffffffffu, m_run, 8 * c);
      const float m1 = __shfl_sync(0xffffffffu, m_run, 8 * c + 4);
      // o[mt][0|2] belong to head 2c, o[mt][1|3] to head 2c+1; dims:
      //   one half (D = 64): o[mt][0|1] -> 8g + 2mt, o[mt][2|3] -> 8g + 2mt + 1
      //   two halves (D = 128): o[mt][0|1] -> 8g + mt, o[mt][2|3] -> 64 + 8g + mt
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int head = 2 * c + j;
        if (head >= G) continue;
        const float lj = j ? l1 : l0;
        const int64_t qrow = static_cast<int64_t>(cons.s) * a.num_q_heads + cons.h * G + head;
        float v[C::HALVES][8];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          if (C::HALVES == 1) {
            v[0][2 * mt] = o[mt][j];
            v[0][2 * mt + 1] = o[mt][2 + j];
          } else {
            v[0][mt] = o[mt][j];
            v[C::HALVES - 1][mt] = o[mt][2 + j];
          }
        }
        if (cons.P_s == 1) {
          const float inv = lj > 0.f ? 1.f / lj : 0.f;
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh) {
            if (a.out_bf16) {
              uint4 w4;
              w4.x = pack_bf16(v[hh][0] * inv, v[hh][1] * inv);
              w4.y = pack_bf16(v[hh][2] * inv, v[hh][3] * inv);
              w4.z = pack_bf16(v[hh][4] * inv, v[hh][5] * inv);
              w4.w = pack_bf16(v[hh][6] * inv, v[hh][7] * inv);
              *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * D + 64 * hh +
                                         8 * g) = w4;
            } else {
              float *dst = static_cast<float *>(a.out) + qrow * D + 64 * hh + 8 * g;
              *reinterpret_cast<float4 *>(dst) =
                  make_float4(v[hh][0] * inv, v[hh][1] * inv, v[hh][2] * inv, v[hh][3] * inv);
              *reinterpret_cast<float4 *>(dst + 4) =
                  make_float4(v[hh][4] * inv, v[hh][5] * inv, v[hh][6] * inv, v[hh][7] * inv);
            }
          }
        } else {
          const int64_t prow = qrow * a.max_partitions + cons.p;
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh) {
            float *dst = a.o_part + prow * D + 64 * hh + 8 * g;
            st_global_keep(dst, make_float4(v[hh][0], v[hh][1], v[hh][2], v[hh][3]), keep_policy);
            st_global_keep(dst + 4, make_float4(v[hh][4], v[hh][5], v[hh][6], v[hh][7]), keep_policy);
          }
          if (g == 0) {
            a.m_part[prow] = j ? m1 : m0;
            a.l_part[prow] = lj;
          }
        }
      }
      // the next record.  The copies in flight are topped up first: items
      // without pages take no stage, so fewer than ST may be in flight, and
      // the producer may still be on this item; topping up records the next.
      ++n_cons_item;
      while (n_issued - n_consumed < ST && issue_next()) {
      }
      cons_enter();
    }
  }
  if constexpr (DYN) {
    if (!left) leave();  // after a timeout
    if (lane == 0) ctl_close(a.ctl, ticket, total_warps, err);
  }
}

// Stage-ring depth: about 12 KiB of pages per warp, at least 2 stages.
template <int D>
constexpr int mma_stages() {
  constexpr int st = (12 * 1024) / (2 * kBlockSize * D * 2);
  return st < 2 ? 2 : st;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder();

// Tensor maps of a cache pool seen as num_rows rows of D bf16 values, 128-byte
// swizzle, one page (16 rows) per box:
//   K: D = 64 -> 2-D {64, rows}, box {64, 16};
//      D = 128 -> 3-D {64, 2, rows}, box {64, 2, 16} (a page lands as [16][128]);
//   V: 2-D {D, rows}, box {64, 16}: one copy per 64-value half.
inline cudaError_t make_page_map(CUtensorMap *map, const void *base, int64_t num_rows, int D,
                                 bool v_halves) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (D == 64 || v_halves) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, kBlockSize};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(num_rows)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(D / 64), kBlockSize};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// L2 lookahead distance for one launch.  Measured on GB300 (same-box
// interleaved runs, inputs not in L2): looking one ring (ST pages) ahead
// shortens long steps (256 sequences of up to 32k tokens: 1.45 -> 1.35 ms;
// the 64-sequence Qwen3 batch with 128-token partitions: 99 -> 94.5 us), and
// longer distances lose (re-reads once the prefetched pages approach L2's
// size).  It is on when the step's page count bound -- sequences x
// ceil(max context / block) x KV heads -- reaches kLookaheadMinPagesPerWarp
// per resident warp; steps below that (tens of pages per warp) lose more at
// start-up than they gain.
constexpr int64_t kLookaheadMinPagesPerWarp = 64;

// Page-balanced pieces for decode steps with a workspace (split-K at all),
// while the unit stream's bound fits the kernels' 32-bit unit arithmetic.
// (Every grid holds at least one warp per KV head: min(items, SMs x CTAs x
// warps) with items >= H_kv and SMs >= H_kv.)
inline bool balanced_pieces(const DecodeArgs &a) {
  if (a.row_of_seq != nullptr || a.seg_count == nullptr) return false;
  const int64_t units = static_cast<int64_t>(a.num_seqs) *
                        ((static_cast<int64_t>(a.ctx_cap) + kBlockSize - 1) / kBlockSize + 1);
  return units <= INT32_MAX / 2;
}

inline int l2_lookahead_pages(const DecodeArgs &a, int64_t warps, int ring_pages) {
  if (a.row_of_seq != nullptr || warps <= 0) return 0;  // prefill: one short item per token
  const int64_t pages = static_cast<int64_t>(a.num_seqs) *
                        ((static_cast<int64_t>(a.ctx_cap) + kBlockSize - 1) / kBlockSize) *
                        a.num_kv_heads;
  return pages >= kLookaheadMinPagesPerWarp * warps ? ring_pages : 0;
}

// d 128 on long steps: 2 warps per CTA with 3 stages of 8 KiB pages (4 CTAs,
// 8 warps per SM; the default is 4 warps with 2 stages, 3 CTAs, 12 warps).
// Measured on GB300 (ragged batches of lognormal(1500, 0.8) contexts, 16/8
// heads, 128-token partitions, inputs not in L2): 128 sequences 0.856 ->
// 0.895 of the copy peak, 256: 0.866 -> 0.951, 384: 0.874 -> 0.966; at 64-96
// sequences the shallower ring with more warps is as fast or faster (0.80 /
// 0.855 vs 0.81 / 0.845; the 64-sequence Qwen3 batch 0.84 vs 0.81).  Chosen
// when the page bound (as for the lookahead) reaches kDeepRingMinPagesPerWarp
// per warp of the deep grid.
constexpr int64_t kDeepRingMinPagesPerWarp = 320;

inline bool deep_ring_preferred(const DecodeArgs &a) {
  if (a.row_of_seq != nullptr) return false;
  const int64_t pages = static_cast<int64_t>(a.num_seqs) *
                        ((static_cast<int64_t>(a.ctx_cap) + kBlockSize - 1) / kBlockSize) *
                        a.num_kv_heads;
  return pages >= kDeepRingMinPagesPerWarp * 8 * device_sm_count();
}

template <int D, int G, int NW, int ST, bool DYN>
cudaError_t launch_mma_kern(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  using C = MmaCfg<D, G, NW, ST>;
  auto kern = paged_decode_mma_kernel<D, G, NW, ST, DYN>;
  static std::atomic<int> occupancy[64];  // per device; 0 = not set up (races recompute it)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (occupancy[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NW * 32, C::SMEM);
    if (e != cudaSuccess) return e;
    occupancy[dev].store(occ > 0 ? occ : 1, std::memory_order_relaxed);
  }
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  e = make_page_map(&tk, a.k_cache, rows, D, false);
  if (e != cudaSuccess) return e;
  e = make_page_map(&tv, a.v_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads;
  const int64_t warps_cap = static_cast<int64_t>(device_sm_count()) *
                            occupancy[dev].load(std::memory_order_relaxed) * NW;
  const int64_t warps = items < warps_cap ? items : warps_cap;
  const int grid = static_cast<int>((warps + NW - 1) / NW);
  if (grid == 0) return cudaSuccess;
  DecodeArgs la = a;
  la.l2_lookahead = l2_lookahead_pages(a, static_cast<int64_t>(grid) * NW, ST);
  la.balanced = 0;
  // Programmatic launch: the grid's CTAs start behind the preceding kernel
  // (the step's write) and run the prologue before griddepcontrol.wait.  In
  // the fixed order a full persistent grid is launched without it: it must
  // find the GPU empty, or CTAs placed late (behind a predecessor's tail)
  // stretch the end of the kernel by a whole CTA's share of the work.  A grid
  // smaller than one wave (a short step: every warp has a single item), and
  // any grid in the dynamic order, launch programmatically.
  if (warps < warps_cap) {
    // about one item per warp: a dynamic order has nothing to even out
    if constexpr (DYN) return launch_mma_kern<D, G, NW, ST, false>(a, err, stream);
    return launch_pdl(kern, dim3(grid), dim3(NW * 32), C::SMEM, stream, tk, tv, la, err);
  }
  // with the dynamic order a CTA placed late only claims fewer items
  if constexpr (DYN) return launch_pdl(kern, dim3(grid), dim3(NW * 32), C::SMEM, stream, tk, tv, la, err);
  kern<<<grid, NW * 32, C::SMEM, stream>>>(tk, tv, la, err);
  return cudaGetLastError();
}

// The bf16 kernel keeps fixed partitions, claimed in dynamic order when the
// call has a workspace.  Page-balanced pieces (which the FP8 kernel takes)
// measured slower here on the same GPU: Qwen3-shape d 128 batches of 64 /
// 128 / 256 / 512 sequences 0.843 -> 0.73, 0.893 -> 0.85, 0.948 -> 0.89,
// 0.977 -> 0.90 of the copy peak (1, 2 or 4 chunks per group no better), the
// long-context d 64 step 0.907 -> 0.921.
template <int D, int G, int NW, int ST>
cudaError_t launch_mma_cfg(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  // the control block's counts have kCtlCountBits bits: claims <= items + warps
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads;
  if (a.ctl && items < (int64_t{1} << (kCtlCountBits - 1)))
    return launch_mma_kern<D, G, NW, ST, true>(a, err, stream);
  return launch_mma_kern<D, G, NW, ST, false>(a, err, stream);
}

template <int D, int G>
cudaError_t launch_mma(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  if constexpr (D == 128) {
    if (deep_ring_preferred(a)) return launch_mma_cfg<D, G, 2, 3>(a, err, stream);
  }
  return launch_mma_cfg<D, G, 4, mma_stages<D>()>(a, err, stream);
}

template <int D>
cudaError_t dispatch_mma_group(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_mma<D, 1>(a, err, stream);
    case 2: return launch_mma<D, 2>(a, err, stream);
    case 4: return launch_mma<D, 4>(a, err, stream);
    case 8: return launch_mma<D, 8>(a, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
