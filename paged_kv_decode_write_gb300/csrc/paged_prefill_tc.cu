// Paged prefill on the fifth-generation tensor cores (tcgen05, TMEM) for
// long prompts: bf16 KV, head_dim 64 or 128, G = H_q / H_kv in {1, 2, 4, 8}.
//
// It computes the prefill definition of photon_paged_attention_prefill: every
// query token of a newly admitted prompt (PhotonInfer README, "Technical
// details > Continuous batching scheduler") attends causally to its
// sequence's tokens 0 .. its position, read through the block table ("Paged
// attention"), with a numerically stable softmax ("Key features >
// GPU-optimised kernels").  Organisation:
//
//  * A row tile is 128 rows: R = 128 / G consecutive query tokens x the G
//    query heads of one KV head (row r = token * G + head).  A work item is
//    one row tile and one KV head; its tokens fall into runs of one sequence
//    ("segments", normally one per tile), each processed over that
//    sequence's keys 0 .. the segment's largest position, with no split: the
//    item writes final output rows.  One CTA of 320 threads per SM walks its
//    items: longest first in a serpentine over the CTAs when it has few
//    items, last first otherwise.
//  * Warp roles.  A producer warp reads the item's token metadata, loads the
//    Q tile by a 3-D TMA tensor copy and the K and V pages of every key tile
//    (128 keys, 8 pages) by 2-D TMA copies into 128-byte-swizzled tiles of
//    64 head dims, in a ring of stages (d 128: K and V of a stage arrive and
//    are released separately), with block-table windows of 32 pages loaded
//    warp-wide.  One lane of an MMA warp issues S = Q K^T into one of NB TMEM
//    buffers (M 128, N 128 keys, K head_dim), ahead of the softmax, and
//    O_h += P_h V_h for each half h of the keys as soon as that half of P is
//    written.  Eight softmax warps hold two threads per row, one per half of
//    the keys: each reads its 64 scores from TMEM, masks (causal, and pages
//    not loaded; only on tiles that need it), keeps a lazy running maximum
//    (moved when passed by more than 8 in base-2 units), and writes its
//    probabilities back
//    into the same TMEM buffer as bf16 pairs P = P_hi + P_lo (both
//    truncations; the P V takes two MMAs and keeps ~16 significant bits),
//    rescaling its half's output accumulator O_h in TMEM only when its
//    maximum moved.
//  * At the end of a segment the two halves combine: out = (f_0 O_0 + f_1 O_1)
//    / (f_0 l_0 + f_1 l_1) with f_h = 2^(m_h - M); each thread stores half of
//    the row's columns (fp32 or bf16).
//  * Every wait is bounded; a timeout sets PHOTON_DEVERR_WAIT_TIMEOUT, the CTA
//    lets its copies land, frees its TMEM and returns.
#include <atomic>
#include <climits>

#include "paged_decode_mma.cuh"
#include "tcgen05.cuh"

namespace photon {
namespace {

constexpr int kTcRows = 128;                        // M: rows of a tile
constexpr int kTcKeys = 128;                        // keys per key tile
constexpr int kTcTilePages = kTcKeys / kBlockSize;  // 8
constexpr int kTcChunk = 128 * 128;                 // one [128 rows][64] bf16 tile: 16 KiB
constexpr int kTcConsumers = 256;                   // 8 softmax warps: two threads per row
constexpr int kTcProducerWarp = kTcConsumers / 32;  // warp 8: loads
constexpr int kTcMmaWarp = kTcProducerWarp + 1;     // warp 9: MMA issue
constexpr int kTcThreads = kTcConsumers + 64;

template <int D>
struct TcCfg {
  static constexpr int CH = D / 64;                  // 64-wide chunks of head_dim
  static constexpr int HALF = D / 2;                 // output columns per thread
  static constexpr int Q_BYTES = CH * kTcChunk;      // a Q tile: CH chunks [128 rows][64]
  static constexpr int Q_OFF = 0;                    // two Q tiles (items in flight)
  static constexpr int KV_OFF = 2 * Q_BYTES;         // stage s: K (CH chunks) then V (CH chunks)
  static constexpr int ST = D == 64 ? 5 : 2;         // ring of key-tile stages
  static constexpr int STAGE = 2 * CH * kTcChunk;
  static constexpr int DATA = KV_OFF + ST * STAGE;
  static constexpr int SMEM = DATA + 1024;           // + 1 KiB alignment slack
  static constexpr int PAGE_TX = CH * kBlockSize * 128;  // K (or V) bytes of one page
  // TMEM columns: NB S buffers (fp32, 128 keys) that then hold that tile's P
  // as bf16 pairs: half h of the keys (keys 64 h .. 64 h + 63) keeps its
  // P_hi in columns 64 h .. 64 h + 31 and its P_lo in 64 h + 32 .. 64 h + 63,
  // i.e. only over its own scores (the other half may not have read its
  // scores yet); then two output accumulators O_0, O_1 (fp32, D dims): one
  // per half of the keys
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NB = (512 - 2 * D) / 128;  // 3 at d 64, 2 at d 128
  static constexpr uint32_t O_COL = 128 * NB;     // O_h at O_COL + h * D
};

// Batches with few items per CTA (fewer than kTcSortMaxItemsPerCta) and at
// most kTcSortMaxTiles row tiles are scheduled longest first: the CTAs rank
// every tile by its key tiles (from its largest position) and take items in a
// serpentine over that order.  Others walk items last first, which with many
// items per CTA is already balanced (8 x 2048-token prompts, same box: with
// ~13 items per CTA (d 128) the sorted order took 400 -> 379 us; with ~27
// (d 64) it cost 448 -> 467 us).
constexpr int kTcSortMaxTiles = 1024;
constexpr int kTcSortMaxItemsPerCta = 16;

// A row's probabilities are taken against a running maximum that is moved
// only when the row maximum exceeds it by more than this (base-2 units), so
// that O rarely needs rescaling; weights stay below 2^kLazyMax.
constexpr float kLazyMax = 8.f;

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int row,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(row), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic: one instruction for two
// lanes of a 64-bit register pair) and the three-input maximum.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Barrier 1 among the 256 softmax threads (the producer warp does not take
// part); the _or form also returns whether any of them passed true.
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool consumer_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

template <int D, int G, bool SORTED>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_q, const DecodeArgs a,
                            int num_items, unsigned int *err) {
  using C = TcCfg<D>;
  constexpr int R = kTcRows / G;  // query tokens per tile
  constexpr int NB = C::NB;
  extern __shared__ unsigned char smem_raw[];
  // With a two-stage ring (d 128) K and V of a stage arrive and are released
  // separately: a K slot is free once its S is computed, about a tile before
  // the V slot, and V trails K by a tile.  Deeper rings (d 64) load both on
  // kfull and release both on kempty after the P V.
  constexpr bool kSplitKV = C::ST <= 2;
  __shared__ __align__(8) uint64_t kfull[C::ST], vfull[C::ST], kempty[C::ST], vempty[C::ST];
  __shared__ __align__(8) uint64_t s_full[NB], p_full[2][NB], pv_done[2][NB];
  __shared__ __align__(8) uint64_t o_free, q_full[2], q_empty[2];
  __shared__ uint32_t page_ok[C::ST];  // pages loaded, per ring stage (producer)
  __shared__ uint32_t page_ok_s[NB];   // the same, per S buffer (MMA warp, for the softmax)
  __shared__ uint32_t tmem_base;
  // per item in flight (two slots): its tokens' sequence rows (-1 none, -2 an
  // out-of-range row) and positions (-1: empty context), its runs of one
  // sequence [seg_start, seg_end) with their contexts
  __shared__ int tok_seq[2][R], tok_pos[2][R];
  __shared__ int seg_start[2][R], seg_end[2][R], seg_ctx[2][R];
  __shared__ int num_segs[2];
  __shared__ float red_m[2][kTcRows], red_l[2][kTcRows];
  __shared__ int tile_cost[SORTED ? kTcSortMaxTiles : 1], tile_of_rank[SORTED ? kTcSortMaxTiles : 1];
  __shared__ volatile int abort_flag;

  const uint32_t raw = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.num_kv_heads, Hq = a.num_q_heads;

  // zeroed stages: pages skipped below (past the context, bad block ids) are
  // masked, and their stale bytes stay finite
  for (int i = tid; i < (C::DATA - C::KV_OFF) / 16; i += kTcThreads)
    reinterpret_cast<uint4 *>(smem + C::KV_OFF)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&s_full[i], 2);  // the S commit and the MMA warp's own arrive
      for (int hf = 0; hf < 2; ++hf) {
        mbar_init(&p_full[hf][i], kTcConsumers / 2);
        mbar_init(&pv_done[hf][i], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(&o_free, 1);
    fence_mbar_init();
    abort_flag = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_q) : "memory");
  }
  fence_proxy_async_smem();
  if (warp == 0) tc::alloc(&tmem_base, C::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_base;
  pdl_launch_dependents();
  pdl_wait();

  // ---- the item order.  Longest first for batches of up to kTcSortMaxTiles
  // tiles: every CTA ranks the tiles the same way (key tiles of the tile's
  // largest valid position, ties by tile index) and item i of that order
  // (tile rank i / H_kv, head i % H_kv) goes to CTA i % grid, forwards in even
  // rounds and backwards in odd ones; larger batches walk items last first.
  const int num_tiles = (a.num_seqs + R - 1) / R;
  constexpr bool sorted = SORTED;  // chosen by the launcher (tc_sorted_order)
  if (sorted) {
    // largest valid position per tile (coalesced reads, shared-memory maxima),
    // then the tile's key tiles (of context that position + 1; 0 if none)
    for (int t = tid; t < num_tiles; t += kTcThreads) tile_cost[t] = -1;
    __syncthreads();
#pragma unroll 4
    for (int tok = tid; tok < a.num_seqs; tok += kTcThreads) {
      const int sq = a.row_of_seq[tok];
      const int ps = a.query_positions[tok];
      if (sq >= 0 && sq < a.num_table_rows && ps >= 0) atomicMax(&tile_cost[tok / R], min(ps, a.ctx_cap - 1));
    }
    __syncthreads();
    for (int t = tid; t < num_tiles; t += kTcThreads) tile_cost[t] = (tile_cost[t] + kTcKeys) / kTcKeys;
    __syncthreads();
    for (int t = tid; t < num_tiles; t += kTcThreads) {
      const int ct = tile_cost[t];
      int rank = 0;
      for (int u = 0; u < num_tiles; ++u) {
        const int cu = tile_cost[u];
        rank += (cu > ct || (cu == ct && u < t)) ? 1 : 0;
      }
      tile_of_rank[rank] = t;
    }
    __syncthreads();
  }
  // the k-th item of this CTA, or false past its last
  auto item_at = [&](int kk, int &tile, int &hh) -> bool {
    if (sorted) {
      const int i = kk * static_cast<int>(gridDim.x) +
                    ((kk & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                              : static_cast<int>(blockIdx.x));
      if (i >= num_items) return false;
      tile = tile_of_rank[i / Hkv];
      hh = i - (i / Hkv) * Hkv;
    } else {
      const int it = static_cast<int>(blockIdx.x) + kk * static_cast<int>(gridDim.x);
      if (it >= num_items) return false;
      const int item = num_items - 1 - it;
      tile = item / Hkv;
      hh = item - tile * Hkv;
    }
    return true;
  };

  if (warp == kTcProducerWarp) {
    // ================= producer warp: item metadata, Q tiles and the K/V
    // ring, running ahead of the other warps
    uint32_t g = 0;
    int k = 0;
    // loop decisions are the warp's, from lane 0 (the lanes shuffle together)
    auto stop_all = [&]() -> bool { return __shfl_sync(0xffffffffu, abort_flag != 0, 0); };
    // lane 0: the V copies of the last tile whose K went out (rows of its
    // pages in the pool view, -1 for pages not loaded)
    bool pend = false;
    uint32_t pend_g = 0;
    int pend_row[kTcTilePages];
    auto issue_v = [&]() -> bool {
      const int st = static_cast<int>(pend_g % C::ST);
      if (pend_g >= C::ST &&
          !mbar_wait_bounded(&vempty[st], ((pend_g / C::ST) - 1) & 1u, kWaitBudgetCycles))
        return false;
      int np = 0;
#pragma unroll
      for (int q = 0; q < kTcTilePages; ++q) np += pend_row[q] >= 0;
      const uint32_t vdst = sbase + C::KV_OFF + st * C::STAGE + C::CH * kTcChunk;
      mbar_arrive_expect_tx(&vfull[st], static_cast<uint32_t>(np * C::PAGE_TX));
#pragma unroll
      for (int q = 0; q < kTcTilePages; ++q) {
        if (pend_row[q] < 0) continue;
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_2d(vdst + c * kTcChunk + q * 2048, &tm_v, 64 * c, pend_row[q], &vfull[st]);
      }
      return true;
    };
    for (;; ++k) {
      int tile, h;
      if (!item_at(k, tile, h) || stop_all()) break;
      const int t0 = tile * R;
      const int slot = k & 1;
      bool ok = true;
      if (lane == 0 && k >= 2)
        ok = mbar_wait_bounded(&q_empty[slot], ((k >> 1) - 1) & 1u, kWaitBudgetCycles);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) abort_flag = 1;
        break;
      }
      for (int r = lane; r < R; r += 32) {
        const int t = t0 + r;
        int seq = -1, pos = -1;
        if (t < a.num_seqs) {
          seq = a.row_of_seq[t];
          pos = a.query_positions[t];
          if (seq < 0 || seq >= a.num_table_rows) {
            atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
            seq = -2;
          } else if (pos >= a.ctx_cap) {
            atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
            pos = a.ctx_cap - 1;
          }
          if (pos < 0) pos = -1;
        }
        tok_seq[slot][r] = seq;
        tok_pos[slot][r] = pos;
      }
      __syncwarp();
      if (lane == 0) {
        // runs of consecutive tokens of one valid sequence
        int n = 0;
        for (int r = 0; r < R;) {
          const int s = tok_seq[slot][r];
          if (s < 0) {
            ++r;
            continue;
          }
          int ctx = 0, e = r;
          while (e < R && tok_seq[slot][e] == s) ctx = max(ctx, tok_pos[slot][e++] + 1);
          seg_start[slot][n] = r;
          seg_end[slot][n] = e;
          seg_ctx[slot][n] = ctx;
          ++n;
          r = e;
        }
        num_segs[slot] = n;
        // the Q tile: rows (token, head) of KV head h (tokens past the end
        // read as zeros); the metadata above is published by the arrive
        mbar_arrive_expect_tx(&q_full[slot], C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          tma_3d(sbase + C::Q_OFF + slot * C::Q_BYTES + c * kTcChunk, &tm_q, 64 * c, h * G, t0,
                 &q_full[slot]);
      }
      __syncwarp();
      // ---- the K/V tiles of every run, the whole warp: lane l holds the
      // block-table entry of page 32 w + l of the run in window w (the next
      // window is loaded while the current one is issued); lane 0 copies, K
      // of a tile before V of the previous tile
      const int n = num_segs[slot];
      bool stop = false;
      for (int sg = 0; sg < n && !stop; ++sg) {
        const int ctx = seg_ctx[slot][sg];
        const int32_t *bt =
            a.block_tables + static_cast<int64_t>(tok_seq[slot][seg_start[slot][sg]]) * a.max_blocks_per_seq;
        auto window = [&](int w) {  // entry of page 32 w + lane, -1 if none or bad
          const int pg = 32 * w + lane;
          int bk = -1;
          if (pg * kBlockSize < ctx) {
            bk = bt[pg];
            if (bk < 0 || bk >= a.num_blocks) {
              atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
              bk = -1;
            }
          }
          return bk;
        };
        int cur = window(0), nxt = 0;
        for (int j = 0; j * kTcKeys < ctx; ++j, ++g) {
          if ((j & 3) == 0) {
            if (j > 0) cur = nxt;
            nxt = (j + 4) * kTcKeys < ctx ? window(j / 4 + 1) : -1;
          }
          const int st = static_cast<int>(g % C::ST);
          int blk[kTcTilePages];
#pragma unroll
          for (int q = 0; q < kTcTilePages; ++q) blk[q] = __shfl_sync(0xffffffffu, cur, (j & 3) * 8 + q);
          bool got = true;
          if (lane == 0) {
            got = abort_flag == 0 &&
                  (g < C::ST || mbar_wait_bounded(&kempty[st], ((g / C::ST) - 1) & 1u, kWaitBudgetCycles));
            if (got) {
              uint32_t mask = 0;
#pragma unroll
              for (int q = 0; q < kTcTilePages; ++q) mask |= (blk[q] >= 0 ? 1u : 0u) << q;
              page_ok[st] = mask;
              const uint32_t kdst = sbase + C::KV_OFF + st * C::STAGE;
              const uint32_t vdst = kdst + C::CH * kTcChunk;
              mbar_arrive_expect_tx(&kfull[st],
                                    static_cast<uint32_t>(__popc(mask) * C::PAGE_TX * (kSplitKV ? 1 : 2)));
#pragma unroll
              for (int q = 0; q < kTcTilePages; ++q) {
                if (blk[q] < 0) continue;
                const int row = (blk[q] * Hkv + h) * kBlockSize;
#pragma unroll
                for (int c = 0; c < C::CH; ++c) {
                  tma_2d(kdst + c * kTcChunk + q * 2048, &tm_k, 64 * c, row, &kfull[st]);
                  if (!kSplitKV) tma_2d(vdst + c * kTcChunk + q * 2048, &tm_v, 64 * c, row, &kfull[st]);
                }
              }
              if (kSplitKV) {  // V of the previous tile, then this tile's V waits
                if (pend) got = issue_v();
                pend = true;
                pend_g = g;
#pragma unroll
                for (int q = 0; q < kTcTilePages; ++q)
                  pend_row[q] = blk[q] < 0 ? -1 : (blk[q] * Hkv + h) * kBlockSize;
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            if (lane == 0) abort_flag = 1;
            stop = true;
            break;
          }
        }
      }
      // the item's last V before the producer may wait for a free slot
      bool got = true;
      if (lane == 0 && pend && !stop) got = issue_v();
      if (lane == 0) pend = false;
      if (stop || !__shfl_sync(0xffffffffu, got, 0)) {
        if (lane == 0) abort_flag = 1;
        break;
      }
      __syncwarp();
    }
  } else if (warp == kTcMmaWarp) {
    // ================= MMA warp (lane 0): S of each key tile ahead of the
    // softmax, each half's P V as soon as that half of P is in TMEM
    if (lane == 0) {
      constexpr uint32_t kIdescS = tc::idesc_bf16(kTcRows, kTcKeys, false);
      constexpr uint32_t kIdescO = tc::idesc_bf16(kTcRows, D, true);
      uint32_t g = 0;
      int k = 0, n_seg = 0;
      bool ok = true;
      // P V of ring tile gg: for each half hf of the keys, O_hf (+)= P_hf V_hf
      // (P = P_hi + P_lo from TMEM buffer gg % NB, columns 64 hf .., rows =
      // lanes, bf16 pairs of keys per column; V rows 64 hf ..), once that half
      // of P is written; then the stage is released
      auto issue_o = [&](uint32_t gg, bool first) -> bool {
        if (kSplitKV && !mbar_wait_bounded(&vfull[gg % C::ST], (gg / C::ST) & 1u, kWaitBudgetCycles))
          return false;
        const uint32_t vb = sbase + C::KV_OFF + (gg % C::ST) * C::STAGE + C::CH * kTcChunk;
        const uint32_t pb = tm + 128 * (gg % NB);
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait_bounded(&p_full[hf][gg % NB], (gg / NB) & 1u, kWaitBudgetCycles)) return false;
          if (hf == 0 && first && n_seg > 0 &&  // O read out by the previous segment
              !mbar_wait_bounded(&o_free, (n_seg - 1) & 1u, kWaitBudgetCycles))
            return false;
          tc::fence_after_sync();
          const uint32_t od = tm + C::O_COL + hf * D;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t vd = tc::desc_sw128(vb + (64 * hf + 16 * kk) * 128, kTcChunk, 1024);
            tc::mma_bf16_tmem_a(od, pb + 64 * hf + kk * 8, vd, kIdescO, !first || kk > 0);
            tc::mma_bf16_tmem_a(od, pb + 64 * hf + 32 + kk * 8, vd, kIdescO, true);
          }
          tc::commit(&pv_done[hf][gg % NB]);
        }
        tc::commit(kSplitKV ? &vempty[gg % C::ST] : &kempty[gg % C::ST]);
        return true;
      };
      for (;; ++k) {
        int tile_unused, h_unused;
        if (!item_at(k, tile_unused, h_unused) || !ok || abort_flag) break;
        const int slot = k & 1;
        if (!mbar_wait_bounded(&q_full[slot], (k >> 1) & 1u, kWaitBudgetCycles)) {
          ok = false;
          break;
        }
        const uint32_t qb = sbase + C::Q_OFF + slot * C::Q_BYTES;
        const int nseg = num_segs[slot];
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const int nkt = (seg_ctx[slot][sg] + kTcKeys - 1) / kTcKeys;
          if (nkt == 0) continue;
          const uint32_t g0 = g;
          for (int j = 0; j < nkt && ok; ++j, ++g) {
            // S of tile g into buffer g % NB, once its pages are in and both
            // halves' P V that last read the buffer are done
            const uint32_t par = ((g / NB) - 1) & 1u;
            if (!mbar_wait_bounded(&kfull[g % C::ST], (g / C::ST) & 1u, kWaitBudgetCycles) ||
                (g >= NB && (!mbar_wait_bounded(&pv_done[0][g % NB], par, kWaitBudgetCycles) ||
                             !mbar_wait_bounded(&pv_done[1][g % NB], par, kWaitBudgetCycles)))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            // the tile's page mask goes with its S (the K slot may be
            // reloaded, and its mask rewritten, before the softmax reads it)
            page_ok_s[g % NB] = page_ok[g % C::ST];
            const uint32_t kb = sbase + C::KV_OFF + (g % C::ST) * C::STAGE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kTcChunk + (kk & 3) * 32;
              tc::mma_bf16(tm + 128 * (g % NB), tc::desc_sw128(qb + off, 16, 1024),
                           tc::desc_sw128(kb + off, 16, 1024), kIdescS, kk > 0);
            }
            tc::commit(&s_full[g % NB]);
            if (kSplitKV) tc::commit(&kempty[g % C::ST]);
            mbar_arrive(&s_full[g % NB]);
            if (j > 0 && !issue_o(g - 1, j == 1)) ok = false;
          }
          if (ok && !issue_o(g0 + nkt - 1, nkt == 1)) ok = false;
          ++n_seg;
        }
      }
      if (!ok) abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ================= 8 softmax warps: two threads per row
    const int row = tid & (kTcRows - 1), half = tid >> 7;
    const uint32_t row_tm = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint32_t g = 0;   // key tiles consumed so far (ring position)
    bool bad = false; // a wait of this thread gave up
    bool abort = false;
    auto store_row = [&](int64_t qrow, int c0, const uint32_t (&v)[32], float scale) {
      if (a.out_bf16) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * D + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(
              pack_bf16(__uint_as_float(v[8 * k]) * scale, __uint_as_float(v[8 * k + 1]) * scale),
              pack_bf16(__uint_as_float(v[8 * k + 2]) * scale, __uint_as_float(v[8 * k + 3]) * scale),
              pack_bf16(__uint_as_float(v[8 * k + 4]) * scale, __uint_as_float(v[8 * k + 5]) * scale),
              pack_bf16(__uint_as_float(v[8 * k + 6]) * scale, __uint_as_float(v[8 * k + 7]) * scale));
      } else {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + qrow * D + c0);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k] = make_float4(__uint_as_float(v[4 * k]) * scale, __uint_as_float(v[4 * k + 1]) * scale,
                               __uint_as_float(v[4 * k + 2]) * scale, __uint_as_float(v[4 * k + 3]) * scale);
      }
    };
    auto zero_row = [&](int64_t qrow) {
      uint32_t z[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = 0u;
#pragma unroll
      for (int c0 = 0; c0 < C::HALF; c0 += 32) store_row(qrow, half * C::HALF + c0, z, 0.f);
    };

    int k = 0;
    for (;; ++k) {
      int tile, h;
      if (!item_at(k, tile, h) || abort) break;
      const int t0 = tile * R;
      const int slot = k & 1;
      // ---- the item's metadata (from the producer)
      if (!mbar_wait_bounded(&q_full[slot], (k >> 1) & 1u, kWaitBudgetCycles)) bad = true;
      const int tok = row / G;
      const int64_t qrow = static_cast<int64_t>(t0 + tok) * Hq + h * G + row % G;
      if (tok_seq[slot][tok] == -2) zero_row(qrow);  // an out-of-range sequence row
      const int nseg = num_segs[slot];

      for (int sg = 0; sg < nseg; ++sg) {
        const int r0 = seg_start[slot][sg], r1 = seg_end[slot][sg];
        const int ctx = seg_ctx[slot][sg];
        const int nkt = (ctx + kTcKeys - 1) / kTcKeys;
        const bool in_seg = tok >= r0 && tok < r1;
        const int mypos = in_seg ? tok_pos[slot][tok] : -1;
        if (nkt == 0) {  // empty contexts (no key tiles are loaded): zero rows
          if (in_seg) zero_row(qrow);
          continue;
        }
        // this half's reference maximum (base-2 units) and sum; its own O_half
        float m_use = -INFINITY, l_run = 0.f;
        // the scores of key tile j are loaded from TMEM while tile j - 1's
        // probabilities are being stored (pre: the loads of tile j are issued)
        uint32_t sv[2][32];
        bool pre = false;
        for (int j = 0; j < nkt; ++j, ++g) {
          if (bad) continue;  // a wait gave up: skip to the segment's end
          const uint32_t b = g % NB;
          const uint32_t buf = row_tm + 128 * b;
          // ---- scores of key tile j (TMEM buffer b); the tile's pages
          if (!pre) {
            if (!mbar_wait_bounded(&s_full[b], (g / NB) & 1u, kWaitBudgetCycles)) {
              bad = true;
              continue;
            }
            tc::fence_after_sync();
            tc::ld32(buf + 64 * half, sv[0]);
            tc::ld32(buf + 64 * half + 32, sv[1]);
          }
          pre = false;
          const uint32_t ok_pages = page_ok_s[b];
          const int kbase = j * kTcKeys;
          if (j == nkt - 1 && (ctx & (kBlockSize - 1)) != 0 &&
              ((ok_pages >> ((ctx - kbase) / kBlockSize)) & 1u)) {
            // slots past the context in the last page may hold any bits:
            // their V rows (weight 0) are zeroed so that 0 * V stays 0 (each
            // half its own keys, once V is in, before it hands its P over)
            if (kSplitKV && !mbar_wait_bounded(&vfull[g % C::ST], (g / C::ST) & 1u, kWaitBudgetCycles)) {
              bad = true;
              continue;
            }
            const int r0z = ctx - kbase, nz = kBlockSize - (ctx & (kBlockSize - 1));
            unsigned char *vt = smem + C::KV_OFF + (g % C::ST) * C::STAGE + C::CH * kTcChunk;
            for (int i = row; i < nz * C::CH * 8; i += kTcRows) {
              const int r = r0z + i / (C::CH * 8), c = (i / 8) % C::CH, v = i % 8;
              if ((r >> 6) == half)
                *reinterpret_cast<uint4 *>(vt + c * kTcChunk + r * 128 + v * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tc::wait_ld();
          tc::pin32(sv[0]);
          tc::pin32(sv[1]);
          // keys visible to this row in the tile: kbase .. min(mypos, kbase + 127);
          // raw scores, masked ones -inf (scale > 0: the maximum of the raw
          // scores gives the maximum of the scaled ones)
          const int nvis = min(max(mypos - kbase + 1, 0), kTcKeys);
          const bool whole = ok_pages == 0xffu && __all_sync(0xffffffffu, nvis == kTcKeys);
          if (!whole) {  // some keys of the tile are hidden from some rows of the warp
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int key = 64 * half + 32 * q + c;
                const bool ok = key < nvis && ((ok_pages >> (key >> 4)) & 1u);
                sv[q][c] = ok ? sv[q][c] : __float_as_uint(-INFINITY);
              }
          }
          // the maximum in four independent chains of three-input maxima
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; c += 8)
#pragma unroll
              for (int t = 0; t < 4; ++t)
                m4[t] = max3(m4[t], __uint_as_float(sv[q][c + 2 * t]), __uint_as_float(sv[q][c + 2 * t + 1]));
          const float mx = max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
          const float m_row = mx * a.scale_log2;
          // move the reference maximum only when this half's maximum passes
          // it by more than kLazyMax (and on the first visible key)
          float m_new = m_use, alpha = 1.f;
          if (m_row > m_use + kLazyMax || (m_use == -INFINITY && m_row != -INFINITY)) {
            m_new = m_row;
            alpha = exp2_approx(m_use - m_new);
          }
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // rescale this row of O_half, once the previous tile's P V of
            // this half is done
            const uint32_t gp = g - 1;
            if (!mbar_wait_bounded(&pv_done[half][gp % NB], (gp / NB) & 1u, kWaitBudgetCycles)) {
              bad = true;
              continue;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ov[32];
              tc::ld32(row_tm + C::O_COL + half * D + c0, ov);
              tc::wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tc::st32(row_tm + C::O_COL + half * D + c0, ov);
            }
          }

          // ---- this thread's 64 probabilities p = 2^(s * scale - m) (a
          // masked -inf gives 0; m kept finite) over its own 64 score columns
          // (read above; the other half's columns may still be unread) as
          // bf16 pairs: P_hi = p truncated to bf16, P_lo = (p - P_hi)
          // truncated (P_hi + P_lo is within 2^-14 of p, relative), keys
          // 64 half + 2c, 2c+1 in column c of each
          const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
          // exponent arguments, sums and remainders two keys per instruction
          // (f32x2); the sums in two independent pairs of accumulators
          const uint64_t scale2 = f32x2(a.scale_log2, a.scale_log2), negm2 = f32x2(neg_m, neg_m);
          uint64_t ls2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float e0, e1;
              unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(sv[q][c]), __uint_as_float(sv[q][c + 1])),
                                     scale2, negm2),
                           e0, e1);
              const float p0 = exp2_approx(e0), p1 = exp2_approx(e1);
              const uint64_t p2 = f32x2(p0, p1);
              ls2[(c >> 1) & 1] = add_f32x2(ls2[(c >> 1) & 1], p2);
              const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
              // p - P_hi with P_hi = p truncated to bf16 (negated: sign bit flipped)
              float d0, d1;
              unpack_f32x2(add_f32x2(p2, f32x2(__uint_as_float((u0 & 0xffff0000u) ^ 0x80000000u),
                                               __uint_as_float((u1 & 0xffff0000u) ^ 0x80000000u))),
                           d0, d1);
              hw[c >> 1] = __byte_perm(u0, u1, 0x7632);
              lw[c >> 1] = __byte_perm(__float_as_uint(d0), __float_as_uint(d1), 0x7632);
            }
            tc::st16(buf + 64 * half + 16 * q, hw);
            tc::st16(buf + 64 * half + 32 + 16 * q, lw);
          }
          float l0a, l0b, l1a, l1b;
          unpack_f32x2(ls2[0], l0a, l0b);
          unpack_f32x2(ls2[1], l1a, l1b);
          const float ls = (l0a + l0b) + (l1a + l1b);
          // the next tile's scores (their own buffer) start loading before this
          // tile's stores are waited for
          if (j + 1 < nkt) {
            const uint32_t gn = g + 1;
            if (mbar_wait_bounded(&s_full[gn % NB], (gn / NB) & 1u, kWaitBudgetCycles)) {
              tc::fence_after_sync();
              tc::ld32(row_tm + 128 * (gn % NB) + 64 * half, sv[0]);
              tc::ld32(row_tm + 128 * (gn % NB) + 64 * half + 32, sv[1]);
              pre = true;
            }  // else the next iteration waits again (and gives up there)
          }
          tc::wait_st();
          l_run = l_run * alpha + ls;
          m_use = m_new;
          tc::fence_before_sync();
          mbar_arrive(&p_full[half][b]);
        }
        // ---- the last P V of this half; then both halves combine: the
        // output row is (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1) with
        // f_h = 2^(m_h - M), M the larger reference; each thread writes half
        // of the row's columns
        if (!bad) {
          const uint32_t gl = g - 1;
          if (!mbar_wait_bounded(&pv_done[half][gl % NB], (gl / NB) & 1u, kWaitBudgetCycles)) bad = true;
        }
        tc::fence_after_sync();
        red_m[half][row] = m_use;
        red_l[half][row] = l_run;
        tc::fence_before_sync();
        if (consumer_sync_or(bad)) {
          abort = true;
          break;
        }
        tc::fence_after_sync();
        const float m0 = red_m[0][row], m1 = red_m[1][row];
        const float M = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.f : exp2_approx(m0 - M);
        const float f1 = m1 == -INFINITY ? 0.f : exp2_approx(m1 - M);
        const float L = red_l[0][row] * f0 + red_l[1][row] * f1;
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < C::HALF; c0 += 32) {
          uint32_t o0[32], o1[32];
          tc::ld32(row_tm + C::O_COL + half * C::HALF + c0, o0);
          tc::ld32(row_tm + C::O_COL + D + half * C::HALF + c0, o1);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            o0[c] = __float_as_uint(__uint_as_float(o0[c]) * f0 + __uint_as_float(o1[c]) * f1);
          if (in_seg) store_row(qrow, half * C::HALF + c0, o0, inv);
        }
        tc::fence_before_sync();
        consumer_sync();  // O and the sums read before the next segment reuses them
        if (tid == 0) mbar_arrive(&o_free);
      }
      if (abort) break;
      // ---- the item's slot (Q tile, metadata) goes back to the producer
      if (consumer_sync_or(bad)) {
        abort = true;
        break;
      }
      if (tid == 0) mbar_arrive(&q_empty[slot]);
    }
    if (abort) abort_flag = 1;
  }
  if (abort_flag) {
    if (tid == 0) atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
    drain_async_copies();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tm, C::TMEM_COLS);
  }
}

// Longest-first order for batches with few items per CTA (see kTcSortMaxTiles).
inline bool tc_sorted_order(int64_t num_tiles, int64_t items, int64_t grid) {
  return num_tiles <= kTcSortMaxTiles && items < kTcSortMaxItemsPerCta * grid;
}

template <int D, int G, bool SORTED>
cudaError_t launch_tc_kernel(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq,
                             const DecodeArgs &a, int grid, int items, unsigned int *err,
                             cudaStream_t stream) {
  using C = TcCfg<D>;
  auto kern = paged_prefill_tc_kernel<D, G, SORTED>;
  static std::atomic<int> ready[64];  // per device: smem attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    ready[dev].store(1, std::memory_order_relaxed);
  }
  kern<<<grid, kTcThreads, C::SMEM, stream>>>(tk, tv, tq, a, items, err);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_tc(DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  cudaError_t e;
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  e = make_page_map(&tk, a.k_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  e = make_page_map(&tv, a.v_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  constexpr int R = kTcRows / G;
  // q viewed as [tokens][H_q][D]: one box is a tile's R tokens x the G query
  // heads of a KV head x 64 dims (rows token * G + head), 128-byte swizzle
  CUtensorMap tq;
  {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(a.num_q_heads),
                                static_cast<cuuint64_t>(a.num_seqs)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(a.num_q_heads) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(R)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t items = (static_cast<int64_t>(a.num_seqs) + R - 1) / R * a.num_kv_heads;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < device_sm_count() ? items : device_sm_count());
  if (grid == 0) return cudaSuccess;
  // every row is written whole: no partitions, nothing for the merge
  a.partition_size = a.ctx_cap > a.partition_size ? a.ctx_cap : a.partition_size;
  const int64_t tiles = (static_cast<int64_t>(a.num_seqs) + R - 1) / R;
  if (tc_sorted_order(tiles, items, grid))
    return launch_tc_kernel<D, G, true>(tk, tv, tq, a, grid, static_cast<int>(items), err, stream);
  return launch_tc_kernel<D, G, false>(tk, tv, tq, a, grid, static_cast<int>(items), err, stream);
}

template <int D>
cudaError_t dispatch_tc(DecodeArgs &a, unsigned int *err, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_tc<D, 1>(a, err, st);
    case 2: return launch_tc<D, 2>(a, err, st);
    case 4: return launch_tc<D, 4>(a, err, st);
    case 8: return launch_tc<D, 8>(a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_tc_preferred(const DecodeArgs &a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  const int64_t tiles = (static_cast<int64_t>(a.num_seqs) + kTcRows / G - 1) / (kTcRows / G);
  return tiles * a.num_kv_heads >= device_sm_count();
}

cudaError_t launch_prefill_tc(DecodeArgs *a, unsigned int *err, cudaStream_t st) {
  switch (a->head_dim) {
    case 64: return dispatch_tc<64>(*a, err, st);
    case 128: return dispatch_tc<128>(*a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
