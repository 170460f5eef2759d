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
//    item writes final output rows.  One CTA of 128 threads per SM walks the
//    items, last first (with tokens in position order the last tiles of a
//    prompt see the most keys).
//  * Per key tile of 128 keys (8 pages): the K and V pages arrive by TMA
//    tensor copies into 128-byte-swizzled tiles of 64 head dims (a ring of
//    stages); thread 0 issues S = Q K^T into TMEM (M 128, N 128, K head_dim;
//    Q and K K-major); every thread then owns one row: it reads its 128
//    scores from TMEM, applies the causal mask (key j visible iff j <= the
//    row's position), updates the running maximum and sum in base 2 and
//    writes its probabilities as bf16 into a swizzled P tile; thread 0 issues
//    O += P V (M 128, N head_dim, K 128 keys; V used MN-major as it lies in
//    the page) into a second TMEM region, then the next tile's S.  When a
//    row's maximum grows, its TMEM output row is rescaled (only warps that
//    need it).
//  * At the end of a segment each thread reads its output row from TMEM,
//    divides by the sum and stores it (fp32 or bf16).
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
constexpr int kTcThreads = 128;

template <int D>
struct TcCfg {
  static constexpr int CH = D / 64;                  // 64-wide chunks of head_dim
  static constexpr int Q_OFF = 0;                    // Q: CH chunks [128 rows][64]
  static constexpr int KV_OFF = CH * kTcChunk;       // stage s: K (CH chunks) then V (CH chunks)
  static constexpr int ST = D == 64 ? 4 : 2;         // ring of key-tile stages
  static constexpr int STAGE = 2 * CH * kTcChunk;
  static constexpr int DATA = KV_OFF + ST * STAGE;
  static constexpr int SMEM = DATA + 1024;           // + 1 KiB alignment slack
  static constexpr int PAGE_TX = 2 * CH * kBlockSize * 128;  // K + V bytes of one page
  // TMEM columns: S (fp32, 128 keys), O (fp32, D dims), P as bf16 pairs in two
  // parts, P = P_hi + P_lo (64 columns each for 128 keys)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0, O_COL = 128, PH_COL = 256, PL_COL = 320;
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int row,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(row), "r"(smem_addr(bar))
      : "memory");
}

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a,
                            int num_items, unsigned int *err) {
  using C = TcCfg<D>;
  constexpr int R = kTcRows / G;  // query tokens per tile
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::ST];
  __shared__ __align__(8) uint64_t s_bar, o_bar;
  __shared__ uint32_t page_ok[C::ST];
  __shared__ uint32_t tmem_base;
  __shared__ int tok_seq[R], tok_pos[R];
  __shared__ int seg_start[R], seg_end[R], seg_seq[R], seg_ctx[R];
  __shared__ int num_segs;

  const uint32_t raw = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int Hkv = a.num_kv_heads, Hq = a.num_q_heads;

  // zeroed stages: pages skipped below (past the context, bad block ids) are
  // masked, and their stale bytes stay finite
  for (int i = tid; i < (C::DATA - C::KV_OFF) / 16; i += kTcThreads)
    reinterpret_cast<uint4 *>(smem + C::KV_OFF)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int i = 0; i < C::ST; ++i) mbar_init(&full_bar[i], 1);
    mbar_init(&s_bar, 1);
    mbar_init(&o_bar, 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
  }
  fence_proxy_async_smem();
  if (warp == 0) tc::alloc(&tmem_base, C::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_base;
  const uint32_t row_tm = tm + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes
  pdl_launch_dependents();
  pdl_wait();

  constexpr uint32_t kIdescS = tc::idesc_bf16(kTcRows, kTcKeys, false);
  constexpr uint32_t kIdescO = tc::idesc_bf16(kTcRows, D, true);
  uint32_t n_tiles = 0;  // key tiles issued so far by this CTA (ring position)
  uint32_t n_s = 0, n_o = 0;  // completed phases of s_bar / o_bar
  bool bad = false;           // this thread saw a wait give up

  // thread 0: starts the copies of key tile j (global tile index g) of
  // sequence seq, KV head h, into its stage; pages at or past ctx are skipped
  auto issue_tile = [&](uint32_t g, int seq, int h, int j, int ctx) {
    const int st = static_cast<int>(g % C::ST);
    const uint32_t kdst = sbase + C::KV_OFF + st * C::STAGE;
    const uint32_t vdst = kdst + C::CH * kTcChunk;
    int blk[kTcTilePages];
    uint32_t mask = 0;
    int n = 0;
    const int32_t *bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
#pragma unroll
    for (int q = 0; q < kTcTilePages; ++q) {
      const int pg = j * kTcTilePages + q;
      blk[q] = -1;
      if (pg * kBlockSize < ctx) {
        const int b = bt[pg];
        if (b >= 0 && b < a.num_blocks) {
          blk[q] = b;
          mask |= 1u << q;
          ++n;
        } else {
          atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
        }
      }
    }
    page_ok[st] = mask;
    mbar_arrive_expect_tx(&full_bar[st], static_cast<uint32_t>(n * C::PAGE_TX));
#pragma unroll
    for (int q = 0; q < kTcTilePages; ++q) {
      if (blk[q] < 0) continue;
      const int row = (blk[q] * Hkv + h) * kBlockSize;
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        tma_2d(kdst + c * kTcChunk + q * 2048, &tm_k, 64 * c, row, &full_bar[st]);
        tma_2d(vdst + c * kTcChunk + q * 2048, &tm_v, 64 * c, row, &full_bar[st]);
      }
    }
  };

  // thread 0: S = Q K^T for the tile in ring position g
  auto issue_s = [&](uint32_t g) {
    const uint32_t kb = sbase + C::KV_OFF + (g % C::ST) * C::STAGE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * kTcChunk + (kk & 3) * 32;
      tc::mma_bf16(tm + C::S_COL, tc::desc_sw128(sbase + C::Q_OFF + off, 16, 1024),
                   tc::desc_sw128(kb + off, 16, 1024), kIdescS, kk > 0);
    }
    tc::commit(&s_bar);
  };

  // thread 0: O (+)= P V for the tile in ring position g, P = P_hi + P_lo
  // from TMEM (rows = lanes, bf16 pairs of keys per column)
  auto issue_o = [&](uint32_t g, bool acc) {
    const uint32_t vb = sbase + C::KV_OFF + (g % C::ST) * C::STAGE + C::CH * kTcChunk;
#pragma unroll
    for (int kk = 0; kk < kTcKeys / 16; ++kk) {
      const uint64_t vd = tc::desc_sw128(vb + kk * 16 * 128, kTcChunk, 1024);
      tc::mma_bf16_tmem_a(tm + C::O_COL, tm + C::PH_COL + kk * 8, vd, kIdescO, acc || kk > 0);
      tc::mma_bf16_tmem_a(tm + C::O_COL, tm + C::PL_COL + kk * 8, vd, kIdescO, true);
    }
    tc::commit(&o_bar);
  };

  bool abort = false;
  for (int it = blockIdx.x; it < num_items && !abort; it += gridDim.x) {
    const int item = num_items - 1 - it;
    const int tile = item / Hkv, h = item - (item / Hkv) * Hkv;
    const int t0 = tile * R;

    // ---- the tile's tokens and their runs of one sequence
    __syncthreads();  // the previous item is done with the token arrays
    if (tid < R) {
      const int t = t0 + tid;
      int seq = -1, pos = -1;
      if (t < a.num_seqs) {
        seq = a.row_of_seq[t];
        pos = a.query_positions[t];
        if (seq < 0 || seq >= a.num_table_rows) {
          atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
          seq = -2;  // a row of zeros
        } else if (pos >= a.ctx_cap) {
          atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
          pos = a.ctx_cap - 1;
        }
        if (pos < 0) pos = -1;
      }
      tok_seq[tid] = seq;
      tok_pos[tid] = pos;
    }
    __syncthreads();
    if (tid == 0) {
      // runs of consecutive tokens of one valid sequence: [seg_start, seg_end)
      int n = 0;
      for (int r = 0; r < R; ++r) {
        const int s = tok_seq[r];
        if (s < 0) continue;
        if (n == 0 || seg_seq[n - 1] != s || seg_end[n - 1] != r) {  // a new run
          seg_start[n] = r;
          seg_seq[n] = s;
          seg_ctx[n] = 0;
          ++n;
        }
        seg_end[n - 1] = r + 1;
        seg_ctx[n - 1] = max(seg_ctx[n - 1], tok_pos[r] + 1);
      }
      num_segs = n;
    }
    // rows of tokens with a bad sequence index are zero rows
    {
      const int tok = tid / G;
      if (tok < R && tok_seq[tok] == -2) {
        const int64_t qrow = static_cast<int64_t>(t0 + tok) * Hq + h * G + tid % G;
        for (int e = 0; e < D; ++e) {
          if (a.out_bf16)
            static_cast<__nv_bfloat16 *>(a.out)[qrow * D + e] = __float2bfloat16_rn(0.f);
          else
            static_cast<float *>(a.out)[qrow * D + e] = 0.f;
        }
      }
    }
    __syncthreads();
    const int nseg = num_segs;

    for (int sg = 0; sg < nseg && !abort; ++sg) {
      const int r0 = seg_start[sg], r1 = seg_end[sg], seq = seg_seq[sg];
      const int ctx = seg_ctx[sg];
      const int nkt = (ctx + kTcKeys - 1) / kTcKeys;
      const int tok = tid / G;
      const bool in_seg = tok >= r0 && tok < r1;
      const int mypos = in_seg ? tok_pos[tok] : -1;
      const int64_t qrow = static_cast<int64_t>(t0 + tok) * Hq + h * G + tid % G;

      if (nkt == 0) {  // empty contexts: zero rows
        if (in_seg)
          for (int e = 0; e < D; ++e) {
            if (a.out_bf16)
              static_cast<__nv_bfloat16 *>(a.out)[qrow * D + e] = __float2bfloat16_rn(0.f);
            else
              static_cast<float *>(a.out)[qrow * D + e] = 0.f;
          }
        continue;
      }

      // ---- Q rows of the segment (others zero) into the swizzled Q tile
      {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) + qrow * D);
#pragma unroll
        for (int e8 = 0; e8 < D / 8; ++e8) {
          const uint4 v = in_seg ? src[e8] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(smem + C::Q_OFF + (e8 >> 3) * kTcChunk +
                                     tc::sw128_offset(tid, (e8 & 7) * 8)) = v;
        }
      }
      fence_proxy_async_smem();
      const uint32_t g0 = n_tiles;
      if (tid == 0)
        for (int j = 0; j < C::ST && j < nkt; ++j) issue_tile(g0 + j, seq, h, j, ctx);
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) {
        if (mbar_wait_bounded(&full_bar[g0 % C::ST], (g0 / C::ST) & 1u, kWaitBudgetCycles)) {
          tc::fence_after_sync();
          issue_s(g0);
        } else {
          bad = true;
        }
      }

      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkt; ++j) {
        const uint32_t g = g0 + j;
        // ---- scores of key tile j
        if (!mbar_wait_bounded(&s_bar, n_s & 1u, kWaitBudgetCycles)) bad = true;
        ++n_s;
        tc::fence_after_sync();
        const uint32_t ok_pages = page_ok[g % C::ST];
        const int kbase = j * kTcKeys;
        if (j == nkt - 1 && (ctx & (kBlockSize - 1)) != 0 &&
            ((ok_pages >> ((ctx - kbase) / kBlockSize)) & 1u)) {
          // slots past the context in the last page may hold any bits: their
          // V rows (weight 0) are zeroed so that 0 * V stays 0
          const int r0z = ctx - kbase, nz = kBlockSize - (ctx & (kBlockSize - 1));
          unsigned char *vt = smem + C::KV_OFF + (g % C::ST) * C::STAGE + C::CH * kTcChunk;
          for (int i = tid; i < nz * C::CH * 8; i += kTcThreads) {
            const int r = r0z + i / (C::CH * 8), c = (i / 8) % C::CH, v = i % 8;
            *reinterpret_cast<uint4 *>(vt + c * kTcChunk + r * 128 + v * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        uint32_t sv[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::ld32(row_tm + 32 * q, sv[q]);
        tc::wait_ld();
        // keys visible to this row in the tile: kbase .. min(mypos, kbase + 127)
        const int nvis = min(max(mypos - kbase + 1, 0), kTcKeys);
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = 32 * q + c;
            const bool ok = key < nvis && ((ok_pages >> (key >> 4)) & 1u);
            const float s = ok ? __uint_as_float(sv[q][c]) * a.scale_log2 : -INFINITY;
            sv[q][c] = __float_as_uint(s);
            mx = fmaxf(mx, s);
          }
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_new == -INFINITY ? 1.f : exp2_approx(m_run - m_new);

        // ---- the previous P V is done (the S commit above covers it): its
        // stage, the P columns and O are free; rescale O rows whose max grew
        if (j > 0) {
          if (!mbar_wait_bounded(&o_bar, n_o & 1u, kWaitBudgetCycles)) bad = true;
          ++n_o;
          tc::fence_after_sync();
          if (tid == 0 && j - 1 + C::ST < nkt) issue_tile(g - 1 + C::ST, seq, h, j - 1 + C::ST, ctx);
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ov[32];
              tc::ld32(row_tm + C::O_COL + c0, ov);
              tc::wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tc::st32(row_tm + C::O_COL + c0, ov);
            }
          }
        }

        // ---- probabilities into TMEM (row = this thread's lane) as bf16
        // pairs, P_hi = bf16(p) and P_lo = bf16(p - P_hi) (about 16
        // significant bits together), keys 2c, 2c+1 in column c
        float ls = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t hw[32], lw[32];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq)
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const int q = 2 * half + qq;
              const float s0 = __uint_as_float(sv[q][c]), s1 = __uint_as_float(sv[q][c + 1]);
              const float p0 = s0 == -INFINITY ? 0.f : exp2_approx(s0 - m_new);
              const float p1 = s1 == -INFINITY ? 0.f : exp2_approx(s1 - m_new);
              ls += p0 + p1;
              const uint32_t w = pack_bf16(p0, p1);
              hw[16 * qq + (c >> 1)] = w;
              lw[16 * qq + (c >> 1)] = pack_bf16(p0 - bf16_lo(w), p1 - bf16_hi(w));
            }
          tc::st32(row_tm + C::PH_COL + 32 * half, hw);
          tc::st32(row_tm + C::PL_COL + 32 * half, lw);
        }
        tc::wait_st();
        l_run = l_run * alpha + ls;
        m_run = m_new;
        tc::fence_before_sync();
        if (__syncthreads_or(bad)) {
          abort = true;
          break;
        }
        tc::fence_after_sync();
        if (tid == 0) {
          issue_o(g, j > 0);
          if (j + 1 < nkt) {
            if (mbar_wait_bounded(&full_bar[(g + 1) % C::ST], ((g + 1) / C::ST) & 1u,
                                  kWaitBudgetCycles)) {
              tc::fence_after_sync();
              issue_s(g + 1);
            } else {
              bad = true;
            }
          }
        }
      }
      if (abort) break;
      n_tiles = g0 + nkt;
      // ---- the last P V: then the output rows
      if (!mbar_wait_bounded(&o_bar, n_o & 1u, kWaitBudgetCycles)) bad = true;
      ++n_o;
      tc::fence_after_sync();
      if (__syncthreads_or(bad)) {
        abort = true;
        break;
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tc::ld32(row_tm + C::O_COL + c0, ov);
        tc::wait_ld();
        if (in_seg) {
          if (a.out_bf16) {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * D + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(
                  pack_bf16(__uint_as_float(ov[8 * v]) * inv, __uint_as_float(ov[8 * v + 1]) * inv),
                  pack_bf16(__uint_as_float(ov[8 * v + 2]) * inv, __uint_as_float(ov[8 * v + 3]) * inv),
                  pack_bf16(__uint_as_float(ov[8 * v + 4]) * inv, __uint_as_float(ov[8 * v + 5]) * inv),
                  pack_bf16(__uint_as_float(ov[8 * v + 6]) * inv, __uint_as_float(ov[8 * v + 7]) * inv));
          } else {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + qrow * D + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(ov[4 * v]) * inv, __uint_as_float(ov[4 * v + 1]) * inv,
                                   __uint_as_float(ov[4 * v + 2]) * inv, __uint_as_float(ov[4 * v + 3]) * inv);
          }
        }
      }
      tc::fence_before_sync();
      __syncthreads();  // O read before the next segment's first P V overwrites it
      tc::fence_after_sync();
    }
  }
  if (abort) {
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

template <int D, int G>
cudaError_t launch_tc(DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  using C = TcCfg<D>;
  auto kern = paged_prefill_tc_kernel<D, G>;
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
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  e = make_page_map(&tk, a.k_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  e = make_page_map(&tv, a.v_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  constexpr int R = kTcRows / G;
  const int64_t items = (static_cast<int64_t>(a.num_seqs) + R - 1) / R * a.num_kv_heads;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < device_sm_count() ? items : device_sm_count());
  if (grid == 0) return cudaSuccess;
  // every row is written whole: no partitions, nothing for the merge
  a.partition_size = a.ctx_cap > a.partition_size ? a.ctx_cap : a.partition_size;
  kern<<<grid, kTcThreads, C::SMEM, stream>>>(tk, tv, a, static_cast<int>(items), err);
  return cudaGetLastError();
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
