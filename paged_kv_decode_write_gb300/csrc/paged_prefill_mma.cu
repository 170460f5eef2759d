// Tiled tensor-core paged prefill for bf16 KV (head_dim 64, 128): causal
// attention of a chunk of query tokens over their sequences' pages, each
// page read once per row tile instead of once per query token.
//
// What it computes is the prefill definition of photon_paged_attention_prefill
// (newly admitted requests write their prompt tokens, PhotonInfer README,
// "Technical details > Continuous batching scheduler"; every such token
// attends causally to its sequence's tokens 0 .. its position), with the
// same online softmax and split-K partial/merge contract as the decode
// kernels.  Organisation:
//
//  * A row tile is R = 16 / G consecutive query tokens.  Its R tokens x G
//    query heads of one KV head fill all 16 rows of the m16n8k16 A operand
//    (row m = token * G + head).  A warp owns whole work items (row tile x
//    KV head x context partition) and its own ring of page stages, with the
//    producer running ahead across items as in the decode kernel.
//  * The tile's tokens fall into runs of one sequence ("segments"; one run in
//    a chunk of a single prompt).  A segment streams its sequence's pages of
//    the partition once for all of its rows; rows of other segments see
//    those pages masked out.
//  * Causal mask: page token j is visible to a row at position p iff j <= p.
//    Pages that every row of a whole-tile segment sees skip the test.
//  * S^T = Q K^T with all 16 rows, online softmax per row, then
//    O^T += V^T P^T over two n-tiles of rows with P from the score fragments
//    (bf16 high part + remainder), as in the decode kernel.  The V^T
//    operand: at head_dim 64 from 16-byte loads and byte permutes (O^T row g
//    of m-tile mt is dim 8g + 2mt, row g+8 dim 8g + 2mt + 1: a lane ends with
//    8 consecutive dims); at head_dim 128 from ldmatrix.trans on the swizzled
//    page (row g is dim 16mt + g, row g+8 dim 16mt + 8 + g), which frees
//    the permute registers: 3 CTAs per SM instead of 2 (8 x 2048-token
//    prompts, Qwen3 heads: 77.6 -> 90.4 TFLOP/s); at 64 the ldmatrix form
//    measured 6 % slower and is not used.
//  * Pages are loaded with the default L2 priority: the other row tiles of
//    the same sequence read them too.
//  * At the end of an item every row whose context fits one partition writes
//    its normalised output; the others write their partial for the merge.
#include <atomic>
#include <climits>
#include <type_traits>

#include "paged_decode_mma.cuh"

namespace photon {
namespace {

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Partitions of a segment whose last position is mx: its context is mx + 1
// (0 for an out-of-range row), at least one partition (which writes the zero
// row of an empty context).
__device__ __forceinline__ int segment_partitions(int seq, int mx, int part) {
  return num_partitions(seq < 0 ? 0 : mx + 1, part);
}

// Position of one warp in its stream of (item, page).  An item is one
// segment (a run of a row tile's tokens in one sequence) x one context
// partition x one KV head; items are numbered segment by segment in token
// order, then partition, then KV head.
struct PfWalker {
  int item;               // global item index
  int cur_tok, cur_base;  // scan cursor: a segment's first token, items before it
  int t0;                 // first query token of the item's row tile
  int r0, r1;             // the item's segment: tile-local tokens [r0, r1)
  int s, minpos;          // its block-table row, smallest position
  int p, h;               // partition, KV head
  int tok1, pg0, n_pages; // pages pg0 .. pg0 + n_pages - 1, tokens below tok1
  int page;               // next page of the item
  bool valid;
};

// Finds w.item with a warp-wide scan over query tokens from the cursor, one
// token per lane: segment starts by ballot (a row-tile boundary or a change
// of sequence), each segment's largest and smallest position by a segmented
// shuffle scan, its items (partitions x KV heads) by a prefix sum.  Only
// segments that end inside the 32-token window count; the cursor then moves
// to the first segment not counted.  Sets w.valid = false past the end.
template <int R>
__device__ __forceinline__ void pf_locate(PfWalker &w, const DecodeArgs &a, int lane) {
  const int H = a.num_kv_heads, part = a.partition_size, T = a.num_seqs;
  w.valid = false;
  while (w.cur_tok < T) {
    const int t = w.cur_tok + lane;
    int seq = -1, pos = -1;
    if (t < T) {
      seq = a.row_of_seq[t];
      pos = a.query_positions[t];
      if (seq < 0 || seq >= a.num_table_rows) seq = -1;
      pos = pos >= a.ctx_cap ? a.ctx_cap - 1 : (pos < 0 ? -1 : pos);
    }
    const int prev = __shfl_up_sync(0xffffffffu, seq, 1);
    const unsigned starts = __ballot_sync(0xffffffffu, t < T && (lane == 0 || t % R == 0 || seq != prev));
    const unsigned upto = lane == 31 ? 0xffffffffu : ((2u << lane) - 1u);
    const int my_start = 31 - __clz(starts & upto);
    int mx = pos, mn = pos;
#pragma unroll
    for (int o = 1; o < R; o <<= 1) {
      const int vx = __shfl_up_sync(0xffffffffu, mx, o);
      const int vn = __shfl_up_sync(0xffffffffu, mn, o);
      if (lane - o >= my_start) {
        mx = max(mx, vx);
        mn = min(mn, vn);
      }
    }
    // a segment ends at this lane if the next token starts one (or is past
    // the end); lane 31 only if the next token begins a row tile
    const bool next_start = lane < 31 ? ((starts >> (lane + 1)) & 1u) != 0 : (t + 1) % R == 0;
    const bool end = t < T && (t + 1 >= T || next_start);
    const int cnt = end ? H * segment_partitions(seq, mx, part) : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, end && w.cur_base + incl > w.item);
    if (hit) {
      const int L = __ffs(hit) - 1;
      const int first = w.cur_base + __shfl_sync(0xffffffffu, incl - cnt, L);
      const int S = __shfl_sync(0xffffffffu, my_start, L);
      const int tL = w.cur_tok + L;
      w.t0 = tL - tL % R;
      w.r0 = w.cur_tok + S - w.t0;
      w.r1 = tL + 1 - w.t0;
      w.s = __shfl_sync(0xffffffffu, seq, L);
      const int smx = __shfl_sync(0xffffffffu, mx, L);
      w.minpos = __shfl_sync(0xffffffffu, mn, L);
      const int off = w.item - first;
      w.p = off / H;
      w.h = off - w.p * H;
      w.cur_tok += S;  // this segment may hold the warp's next item too
      w.cur_base = first;
      const int tok0 = w.p * part;
      w.tok1 = min(tok0 + part, w.s < 0 ? 0 : smx + 1);
      w.pg0 = tok0 / kBlockSize;
      w.n_pages = w.tok1 > tok0 ? (w.tok1 - tok0 + kBlockSize - 1) / kBlockSize : 0;
      w.page = 0;
      w.valid = true;
      return;
    }
    // past the window's last counted segment end (a segment running on past
    // lane 31 is counted in the next window; segments are at most R <= 16
    // tokens, so one always ends in the window)
    const unsigned ends = __ballot_sync(0xffffffffu, end);
    w.cur_base += __shfl_sync(0xffffffffu, incl, 31);
    w.cur_tok += 32 - __clz(ends);
  }
}

// PP pages per pipeline stage and softmax step: a stage holds
// [K page 0] .. [K page PP-1] [V page 0] .. [V page PP-1].
template <int D, int PP>
__host__ __device__ constexpr int prefill_stage_bytes() {
  return 2 * PP * kBlockSize * D * 2;
}

template <int D, int G, int NW, int ST, int PP>
__global__ void __launch_bounds__(NW * 32)
    paged_prefill_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a,
                             unsigned int *err) {
  using C = MmaCfg<D, G, NW, ST>;
  constexpr int R = 16 / G;
  constexpr int SB = prefill_stage_bytes<D, PP>();
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  unsigned char *stages = smem + warp * ST * SB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * ST * SB) + warp * ST;
  const uint32_t stages_s = smem_addr(stages);

  if (lane == 0) {
    for (int i = 0; i < ST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
  }
  __syncwarp();
  pdl_launch_dependents();
  pdl_wait();

  const uint64_t policy = l2_evict_normal_policy();
  const uint64_t keep_policy = l2_evict_last_policy();
  const int total_warps = gridDim.x * NW;

  // fragment offsets inside a stage, as in the decode kernel
  uint32_t koff[2][C::KCH];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < C::KCH; ++i)
      koff[nt][i] = swz128((8 * nt + g) * C::ROW_BYTES + (C::KCH * c + i) * 16);
  uint32_t voff[4][C::HALVES];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int hh = 0; hh < C::HALVES; ++hh) {
      const int row = 2 * c + (r & 1) + 8 * (r >> 1);
      voff[r][hh] = hh * (kBlockSize * 128) + swz128(row * 128 + g * 16);  // within a V page
    }
  // ldmatrix.x4.trans of V^T: lanes 8j .. 8j+7 address rows of matrix j =
  // page tokens (lane & 7) + 8 (j >> 1), dims 8 (j & 1) .. +7 of the m-tile;
  // a 16-byte chunk k of token row t sits at t * 128 + ((k ^ (t & 7)) << 4)
  const int ldm_tok = (lane & 7) + 8 * ((lane >> 4) & 1);
  const uint32_t ldm_row = ldm_tok * 128, ldm_x = ldm_tok & 7, ldm_hi = (lane >> 3) & 1;

  PfWalker prod, cons;
  prod.item = cons.item = blockIdx.x * NW + warp;
  prod.cur_tok = prod.cur_base = cons.cur_tok = cons.cur_base = 0;
  pf_locate<R>(prod, a, lane);
  pf_locate<R>(cons, a, lane);
  uint32_t n_issued = 0, valid_bits = 0;
  uint32_t c_slot = 0, c_phase = 0;
  int bt_base = INT_MIN / 2, bt_reg = -1;

  // Issues the producer's next PP pages (those past the item are skipped).
  auto issue_next = [&]() -> bool {
    while (prod.valid && prod.page >= prod.n_pages) {
      prod.item += total_warps;
      pf_locate<R>(prod, a, lane);
      bt_base = INT_MIN / 2;
    }
    if (!prod.valid) return false;
    if (prod.page + PP - 1 - bt_base >= 32) {
      bt_base = prod.page;
      bt_reg = bt_base + lane < prod.n_pages
                   ? a.block_tables[static_cast<int64_t>(prod.s) * a.max_blocks_per_seq +
                                    prod.pg0 + bt_base + lane]
                   : -1;
    }
    int blk[PP];
#pragma unroll
    for (int pp = 0; pp < PP; ++pp) {
      const int b = __shfl_sync(0xffffffffu, bt_reg, prod.page + pp - bt_base);
      blk[pp] = prod.page + pp < prod.n_pages ? b : INT_MIN;  // INT_MIN: past the item
    }
    const uint32_t st = n_issued % ST;
    if (lane == 0) {
      uint32_t bits = 0, bytes = 0;
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        if (blk[pp] >= 0 && blk[pp] < a.num_blocks) {
          bits |= 1u << pp;
          bytes += 2 * C::PAGE_BYTES;
        } else if (blk[pp] != INT_MIN) {
          atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
        }
      }
      unsigned char *dst = stages + st * SB;
      fence_proxy_async_smem();
      if (bytes) {
        mbar_arrive_expect_tx(&bars[st], bytes);
#pragma unroll
        for (int pp = 0; pp < PP; ++pp)
          if ((bits >> pp) & 1u) {
            const int row = (blk[pp] * a.num_kv_heads + prod.h) * kBlockSize;
            tma_load_k_page<D>(dst + pp * C::PAGE_BYTES, &tm_k, row, &bars[st], policy);
            tma_load_v_page<D>(dst + (PP + pp) * C::PAGE_BYTES, &tm_v, row, &bars[st], policy);
          }
      } else {
        mbar_arrive(&bars[st]);
      }
      valid_bits = (valid_bits & ~(((1u << PP) - 1u) << (PP * st))) | (bits << (PP * st));
    }
    prod.page += PP;
    ++n_issued;
    return true;
  };

  for (int k = 0; k < ST; ++k)
    if (!issue_next()) break;

  // rows g and g + 8 of the tile: tile-local tokens and heads
  const int tg0 = g / G, tg1 = (g + 8) / G;
  uint32_t qa[C::KT][4];     // A fragments: rows g, g+8, permuted head dims
  float o[C::MT][2][4];      // O^T fragments, n-tile n2 = rows 8*n2 .. 8*n2+7
  float m_run[2], l_run[2];  // rows g, g+8 (l: over this lane's tokens)
  int lim[2];                // last visible position of rows g, g+8 (-1: not in the item)
  bool whole = false;        // the item's segment holds every row of the tile
  int cur_item = -1;

  while (cons.valid) {
    if (cons.item != cur_item) {
      // new item: query rows of its segment (bf16 words, permuted head dims),
      // their visibility limits; the tile's other rows stay zero and masked
      cur_item = cons.item;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int tok = half ? tg1 : tg0;
        const int head = (half ? g + 8 : g) % G;
        const bool in = tok >= cons.r0 && tok < cons.r1;
        uint32_t qw[C::KW];
        int lp = -1;
        if (in) {
          const int t = cons.t0 + tok;
          lp = a.query_positions[t];
          if (lp >= a.ctx_cap) {
            atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
            lp = a.ctx_cap - 1;
          }
          if (cons.s < 0) {
            atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
            lp = -1;
          }
          const uint4 *src = reinterpret_cast<const uint4 *>(
              static_cast<const __nv_bfloat16 *>(a.q) +
              (static_cast<int64_t>(t) * a.num_q_heads + cons.h * G + head) * D + C::KW * 2 * c);
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
        lim[half] = lp < 0 ? -1 : lp;
#pragma unroll
        for (int kt = 0; kt < C::KT; ++kt) {
          qa[kt][half] = qw[2 * kt];          // a0 (row g) / a1 (row g+8): k low
          qa[kt][2 + half] = qw[2 * kt + 1];  // a2 / a3: k high
        }
      }
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int n2 = 0; n2 < 2; ++n2) o[mt][n2][0] = o[mt][n2][1] = o[mt][n2][2] = o[mt][n2][3] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
      whole = cons.r0 == 0 && cons.r1 == R;
    }

    if (cons.page < cons.n_pages) {
      const uint32_t st = c_slot;
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], c_phase, kWaitBudgetCycles));
      if (!ok) {
        if (lane == 0) atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
        drain_async_copies();
        return;
      }
      const uint32_t vb = __shfl_sync(0xffffffffu, valid_bits >> (PP * st), 0);
      int ptok[PP], nv[PP];  // first token and valid tokens of each page (0: skipped)
      bool full = whole;
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        ptok[pp] = (cons.pg0 + cons.page + pp) * kBlockSize;
        nv[pp] = ((vb >> pp) & 1u) ? max(0, min(kBlockSize, cons.tok1 - ptok[pp])) : 0;
        full = full && nv[pp] == kBlockSize;
      }
      full = full && cons.minpos >= ptok[PP - 1] + kBlockSize - 1;  // every row sees every token
      const uint32_t base = stages_s + st * SB;
      // ---- S^T = Q K^T per page: rows g (s[pp][nt][0..1]) and g+8 ([2..3]), tokens 8nt + 2c + j
      float s[PP][2][4];
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t kw[C::KW];
#pragma unroll
          for (int i = 0; i < C::KCH; ++i)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(kw[4 * i]), "=r"(kw[4 * i + 1]), "=r"(kw[4 * i + 2]),
                           "=r"(kw[4 * i + 3])
                         : "r"(base + pp * C::PAGE_BYTES + koff[nt][i]));
          s[pp][nt][0] = s[pp][nt][1] = s[pp][nt][2] = s[pp][nt][3] = 0.f;
#pragma unroll
          for (int kt = 0; kt < C::KT; ++kt)
            mma_bf16_16816_full(s[pp][nt], qa[kt][0], qa[kt][1], qa[kt][2], qa[kt][3], kw[2 * kt],
                                kw[2 * kt + 1]);
        }
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) s[pp][nt][j] *= a.scale_log2;
      if (!full) {  // causal and segment mask; skipped pages are wholly masked
#pragma unroll
        for (int pp = 0; pp < PP; ++pp)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (nv[pp] == 0 || ptok[pp] + 8 * nt + 2 * c + (j & 1) > lim[j >> 1])
                s[pp][nt][j] = -INFINITY;
      }
      // ---- online softmax over the stage's PP pages, rows g and g+8
      float alpha[2], mu[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mx = -INFINITY;
#pragma unroll
        for (int pp = 0; pp < PP; ++pp)
          mx = fmaxf(mx, fmaxf(fmaxf(s[pp][0][2 * r], s[pp][0][2 * r + 1]),
                               fmaxf(s[pp][1][2 * r], s[pp][1][2 * r + 1])));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[r], mx);
        mu[r] = m_new == -INFINITY ? 0.f : m_new;  // a row with nothing visible yet
        alpha[r] = exp2_approx(m_run[r] - mu[r]);
        m_run[r] = m_new;
      }
      float ps[2] = {0.f, 0.f};
      uint32_t ph[2][PP][2], pl[2][PP][2];  // [n2][page][nt]: P^T B fragments of row n-tile n2
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float p0 = exp2_approx(s[pp][nt][2 * r] - mu[r]);
            const float p1 = exp2_approx(s[pp][nt][2 * r + 1] - mu[r]);
            ps[r] += p0 + p1;
            ph[r][pp][nt] = pack_bf16(p0, p1);
            pl[r][pp][nt] = pack_bf16(p0 - bf16_lo(ph[r][pp][nt]), p1 - bf16_hi(ph[r][pp][nt]));
          }
      l_run[0] = fmaf(l_run[0], alpha[0], ps[0]);
      l_run[1] = fmaf(l_run[1], alpha[1], ps[1]);
      // O^T columns of this lane: rows 8*n2 + 2c + j, whose alpha sits in lane 8c + 4j
#pragma unroll
      for (int n2 = 0; n2 < 2; ++n2) {
        const float a0 = __shfl_sync(0xffffffffu, alpha[n2], 8 * c);
        const float a1 = __shfl_sync(0xffffffffu, alpha[n2], 8 * c + 4);
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          o[mt][n2][0] *= a0;
          o[mt][n2][1] *= a1;
          o[mt][n2][2] *= a0;
          o[mt][n2][3] *= a1;
        }
      }
      if constexpr (C::HALVES == 1) {
      // ---- O^T += V^T P^T, page by page (skipped pages hold stale bytes: not read)
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        if (nv[pp] == 0) continue;
        const uint32_t vbase = base + (PP + pp) * C::PAGE_BYTES;
        uint32_t vw[4][4 * C::HALVES];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(vw[r][4 * hh]), "=r"(vw[r][4 * hh + 1]), "=r"(vw[r][4 * hh + 2]),
                           "=r"(vw[r][4 * hh + 3])
                         : "r"(vbase + voff[r][hh]));
        if (nv[pp] < kBlockSize) {  // rows past the sequence's last token may hold any bits
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = 2 * c + (r & 1) + 8 * (r >> 1);
            if (row >= nv[pp])
#pragma unroll
              for (int i = 0; i < 4 * C::HALVES; ++i) vw[r][i] = 0u;
          }
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          uint32_t a_0, a_1, a_2, a_3;
          if (C::HALVES == 1) {
            a_0 = __byte_perm(vw[0][mt], vw[1][mt], 0x5410u);
            a_1 = __byte_perm(vw[0][mt], vw[1][mt], 0x7632u);
            a_2 = __byte_perm(vw[2][mt], vw[3][mt], 0x5410u);
            a_3 = __byte_perm(vw[2][mt], vw[3][mt], 0x7632u);
          } else {
            const int ww = mt >> 1;
            const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
            a_0 = __byte_perm(vw[0][ww], vw[1][ww], sel);
            a_1 = __byte_perm(vw[0][4 + ww], vw[1][4 + ww], sel);
            a_2 = __byte_perm(vw[2][ww], vw[3][ww], sel);
            a_3 = __byte_perm(vw[2][4 + ww], vw[3][4 + ww], sel);
          }
#pragma unroll
          for (int n2 = 0; n2 < 2; ++n2) {
            mma_bf16_16816_full(o[mt][n2], a_0, a_1, a_2, a_3, ph[n2][pp][0], ph[n2][pp][1]);
            mma_bf16_16816_full(o[mt][n2], a_0, a_1, a_2, a_3, pl[n2][pp][0], pl[n2][pp][1]);
          }
        }
      }
      } else {
      // ---- O^T += V^T P^T, page by page (skipped pages hold stale bytes: not read)
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        if (nv[pp] == 0) continue;
        const uint32_t vbase = base + (PP + pp) * C::PAGE_BYTES;
        // tokens past the sequence's last one may hold any bits: zero their halves
        uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
        if (nv[pp] < kBlockSize) {
          m01 = (2 * c < nv[pp] ? 0x0000ffffu : 0u) | (2 * c + 1 < nv[pp] ? 0xffff0000u : 0u);
          m23 = (2 * c + 8 < nv[pp] ? 0x0000ffffu : 0u) | (2 * c + 9 < nv[pp] ? 0xffff0000u : 0u);
        }
        auto pv_page = [&](auto masked_tag) {
          constexpr bool masked = decltype(masked_tag)::value;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            // V^T A fragment of dims 16mt .. 16mt+15 straight from the swizzled page
            uint32_t a_0, a_1, a_2, a_3;
            const uint32_t chunk = 2 * (mt & 3) + ldm_hi;
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a_0), "=r"(a_1), "=r"(a_2), "=r"(a_3)
                         : "r"(vbase + (mt >> 2) * (kBlockSize * 128) + ldm_row +
                               ((chunk ^ ldm_x) << 4)));
            if (masked) {
              a_0 &= m01;
              a_1 &= m01;
              a_2 &= m23;
              a_3 &= m23;
            }
#pragma unroll
            for (int n2 = 0; n2 < 2; ++n2) {
              mma_bf16_16816_full(o[mt][n2], a_0, a_1, a_2, a_3, ph[n2][pp][0], ph[n2][pp][1]);
              mma_bf16_16816_full(o[mt][n2], a_0, a_1, a_2, a_3, pl[n2][pp][0], pl[n2][pp][1]);
            }
          }
        };
        if (nv[pp] < kBlockSize)
          pv_page(std::true_type{});
        else
          pv_page(std::false_type{});
      }
      }
      __syncwarp();
      if (++c_slot == ST) {
        c_slot = 0;
        c_phase ^= 1u;
      }
      cons.page += PP;
      issue_next();
    }

    if (cons.page >= cons.n_pages) {
      // ---- item done: the segment's rows whose context reaches partition p
      float lt[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lt[r] = l_run[r];
        lt[r] += __shfl_xor_sync(0xffffffffu, lt[r], 1);
        lt[r] += __shfl_xor_sync(0xffffffffu, lt[r], 2);
      }
#pragma unroll
      for (int n2 = 0; n2 < 2; ++n2)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int row = 8 * n2 + 2 * c + j;  // this lane's O^T column
          const int src_lane = 8 * c + 4 * j;  // holds the row as its row g (n2 0) or g+8 (n2 1)
          const float L = __shfl_sync(0xffffffffu, lt[n2], src_lane);
          const float M = __shfl_sync(0xffffffffu, m_run[n2], src_lane);
          const int lp = __shfl_sync(0xffffffffu, lim[n2], src_lane);
          const int tok = row / G, head = row % G;
          if (tok < cons.r0 || tok >= cons.r1) continue;
          const int P_t = num_partitions(lp + 1, a.partition_size);
          if (cons.p >= P_t) continue;
          const int64_t qrow = static_cast<int64_t>(cons.t0 + tok) * a.num_q_heads + cons.h * G + head;
          if constexpr (C::HALVES == 1) {
          float v[C::HALVES][8];
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            if (C::HALVES == 1) {
              v[0][2 * mt] = o[mt][n2][j];
              v[0][2 * mt + 1] = o[mt][n2][2 + j];
            } else {
              v[0][mt] = o[mt][n2][j];
              v[C::HALVES - 1][mt] = o[mt][n2][2 + j];
            }
          }
          if (P_t == 1) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int hh = 0; hh < C::HALVES; ++hh) {
              if (a.out_bf16) {
                uint4 w4;
                w4.x = pack_bf16(v[hh][0] * inv, v[hh][1] * inv);
                w4.y = pack_bf16(v[hh][2] * inv, v[hh][3] * inv);
                w4.z = pack_bf16(v[hh][4] * inv, v[hh][5] * inv);
                w4.w = pack_bf16(v[hh][6] * inv, v[hh][7] * inv);
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * D +
                                           64 * hh + 8 * g) = w4;
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
              st_global_keep(dst + 4, make_float4(v[hh][4], v[hh][5], v[hh][6], v[hh][7]),
                             keep_policy);
            }
            if (g == 0) {
              a.m_part[prow] = M;
              a.l_part[prow] = L;
            }
          }
          } else {
          // O^T rows of m-tile mt: row g is dim 16mt + g, row g+8 dim 16mt + 8 + g
          // (ldmatrix hands lane g element g of each 16-byte V row); the
          // eight lanes g of a column store 32 contiguous bytes per dim group
          if (P_t == 1) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
              for (int hi = 0; hi < 2; ++hi) {
                const int64_t idx = qrow * D + 16 * mt + 8 * hi + g;
                const float val = o[mt][n2][2 * hi + j] * inv;
                if (a.out_bf16)
                  static_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(val);
                else
                  static_cast<float *>(a.out)[idx] = val;
              }
          } else {
            const int64_t prow = qrow * a.max_partitions + cons.p;
            float *dst = a.o_part + prow * D + g;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
              for (int hi = 0; hi < 2; ++hi)
                asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst + 16 * mt + 8 * hi),
                             "f"(o[mt][n2][2 * hi + j]), "l"(keep_policy)
                             : "memory");
            if (g == 0) {
              a.m_part[prow] = M;
              a.l_part[prow] = L;
            }
          }
          }
        }
      cons.item += total_warps;
      pf_locate<R>(cons, a, lane);
    }
  }
}

// Split-K partitions exist to create work.  When the row tiles alone give
// every resident warp at least two items, the launch merges the caller's
// partitions into ones of about kCoarsePartition tokens (a multiple of the
// caller's size, so the workspace still fits): long prompts then write few
// partials and the merge has little to do.  The result is the same
// mathematically.
constexpr int64_t kCoarsePartition = 4096;

template <int D, int G>
cudaError_t launch_prefill(DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  // d 64: two-page stages, two of them (16 KiB per warp; registers allow 3
  // CTAs per SM anyway); d 128: one-page stages, as in the decode kernel.
  constexpr int NW = 4;
  constexpr int PP = D == 64 ? 2 : 1;
  constexpr int ST = D == 64 ? 2 : mma_stages<D>();
  constexpr int SMEM = NW * ST * prefill_stage_bytes<D, PP>() + NW * ST * 8 + 1024;
  auto kern = paged_prefill_mma_kernel<D, G, NW, ST, PP>;
  static std::atomic<int> occupancy[64];  // per device; 0 = not set up (races recompute it)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (occupancy[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NW * 32, SMEM);
    if (e != cudaSuccess) return e;
    occupancy[dev].store(occ > 0 ? occ : 1, std::memory_order_relaxed);
  }
  const int64_t rows = a.num_blocks * a.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  e = make_page_map(&tk, a.k_cache, rows, D, false);
  if (e != cudaSuccess) return e;
  e = make_page_map(&tv, a.v_cache, rows, D, true);
  if (e != cudaSuccess) return e;
  // at most one segment per query token
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads;
  if (items > INT_MAX) return cudaErrorInvalidValue;
  const int64_t warps_cap = static_cast<int64_t>(device_sm_count()) *
                            occupancy[dev].load(std::memory_order_relaxed) * NW;
  const int64_t tiles = (static_cast<int64_t>(a.num_seqs) + 16 / G - 1) / (16 / G);
  if (tiles * a.num_kv_heads >= 2 * warps_cap && a.partition_size < kCoarsePartition) {
    const int64_t k = (kCoarsePartition + a.partition_size - 1) / a.partition_size;
    a.partition_size = static_cast<int32_t>(k * a.partition_size);
  }
  const int64_t warps = items < warps_cap ? items : warps_cap;
  const int grid = static_cast<int>((warps + NW - 1) / NW);
  if (grid == 0) return cudaSuccess;
  kern<<<grid, NW * 32, SMEM, stream>>>(tk, tv, a, err);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_prefill_group(DecodeArgs &a, unsigned int *err, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_prefill<D, 1>(a, err, st);
    case 2: return launch_prefill<D, 2>(a, err, st);
    case 4: return launch_prefill<D, 4>(a, err, st);
    case 8: return launch_prefill<D, 8>(a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_tiled_supported(const DecodeArgs &a, photon_dtype kv_dtype) {
  const int G = a.num_kv_heads > 0 ? a.num_q_heads / a.num_kv_heads : 0;
  return kv_dtype == PHOTON_BF16 && (a.head_dim == 64 || a.head_dim == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8) &&
         a.num_blocks * a.num_kv_heads * kBlockSize <= INT32_MAX &&
         static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads <= INT32_MAX;
}

cudaError_t launch_prefill_tiled(DecodeArgs *a, unsigned int *err, cudaStream_t st) {
  switch (a->head_dim) {
    case 64: return dispatch_prefill_group<64>(*a, err, st);
    case 128: return dispatch_prefill_group<128>(*a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
