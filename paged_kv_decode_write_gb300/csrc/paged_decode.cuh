// Split-K paged decode attention for sm_103a: the partial kernel (one work
// item = one sequence x one KV head x one context partition) and the
// log-sum-exp merge kernel.
//
// PhotonInfer README, "Key features > GPU-optimised kernels": batched paged
// attention over the block-level cache, vectorised memory access, and a
// numerically stable attention softmax.  The design here is GB300-first:
//
//  * Persistent CTAs (SM count x resident CTAs per SM) walk the work items in
//    a fixed stride.  The (sequence, partition) of an item is found on the
//    device from context_lens with a warp-wide prefix sum over a forward-only
//    cursor, so the host passes no work list and reads nothing back.
//  * Each of the NW warps of a CTA takes every NW-th page of the item and runs
//    its own ST-deep ring of shared-memory stages.  One lane issues, per page,
//    two bulk copies on the TMA engine (the page's K rows and V rows are each
//    one contiguous bs*d run in the [block][kv_head][slot][dim] layout), with
//    an evict-first L2 hint, and an mbarrier completes when the bytes land.
//  * A warp reads a staged page as 16-byte vectors: LPT lanes cover one token
//    row, so 32 lanes read TPI full rows per instruction without bank
//    conflicts.  The query group (G heads sharing the KV head) sits in
//    registers pre-scaled by scale*log2(e); each K vector feeds G dot
//    products, finished by xor-shuffles inside the row's lanes.
//  * Online softmax in base 2 per head: page maximum by shuffles, running
//    max/sum rescaled per page, exp2 of the shifted scores, then the V
//    vectors accumulate into G x E fp32 registers per lane.
//  * At the end of an item the warps merge their (max, sum, output) through
//    shared memory; a single-partition sequence writes its normalised output,
//    otherwise the unnormalised partial and its (max, sum) go to the
//    workspace for the merge kernel.
//  * Every wait is bounded; a block id outside the pool skips that page and a
//    context length beyond the bounds is clamped, both setting a sticky bit.
#pragma once

#include <atomic>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace photon {

template <typename Tag, int D, int G, int NW, int ST>
struct DecodeCfg {
  using T = typename Tag::T;
  static constexpr int E = Unpack<Tag>::kElems;        // elements per 16-byte vector
  static constexpr int LPT = D / E;                    // lanes per token row
  static constexpr int TPI = 32 / LPT;                 // token rows per warp-wide load
  static constexpr int ITERS = kBlockSize / TPI;       // warp-wide loads per page
  static constexpr int PAGE_BYTES = kBlockSize * D * Tag::kBytes;  // K (or V) of one page
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int SMEM_STAGES = NW * ST * STAGE_BYTES;
  static constexpr int SMEM_BARS = NW * ST * 8;
  static constexpr int SMEM_MERGE = NW * G * (D + 2) * 4;
  static constexpr int SMEM_TOTAL = SMEM_STAGES + SMEM_BARS + SMEM_MERGE + 16;
  static_assert(LPT >= 1 && LPT <= 32 && TPI * LPT == 32, "head_dim / vector mismatch");
  static_assert(ITERS * TPI == kBlockSize, "block size must be a multiple of rows per load");
  static_assert(ST >= 1 && ST <= 32, "stage ring");
};

// Roughly 0.2 s at GB300 clocks: far beyond any real page-copy latency.
constexpr long long kWaitBudgetCycles = 400000000LL;

__device__ __forceinline__ int clamp_context(int c, int cap, unsigned int *err) {
  if (c > cap) {
    atomicOr(err, PHOTON_DEVERR_CONTEXT_RANGE);
    return cap;
  }
  return c < 0 ? 0 : c;
}

// Context length of (virtual) sequence s: context_lens[s] for decode, the
// query's position + 1 for prefill.  A prefill token whose table row is out
// of range gets an empty context (and the block-range bit).
__device__ __forceinline__ int seq_context(const DecodeArgs &a, int s, unsigned int *err) {
  if (!a.query_positions) return a.context_lens[s];
  const int row = a.row_of_seq[s];
  if (row < 0 || row >= a.num_table_rows) {
    atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
    return 0;
  }
  return a.query_positions[s] + 1;
}

// Block-table row of (virtual) sequence s (checked by seq_context).
__device__ __forceinline__ int64_t seq_table_row(const DecodeArgs &a, int s) {
  return a.row_of_seq ? a.row_of_seq[s] : s;
}

// Partitions of a sequence: at least one, so an empty context still owns an
// item (which writes its zero output row).
__device__ __forceinline__ int num_partitions(int ctx, int part) {
  return ctx <= 0 ? 1 : (ctx + part - 1) / part;
}

template <typename Tag, int D, int G, int NW, int ST>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_partial_kernel(const DecodeArgs a, unsigned int *err) {
  using C = DecodeCfg<Tag, D, G, NW, ST>;
  using T = typename Tag::T;
  extern __shared__ __align__(128) unsigned char smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int chunk = lane % C::LPT;  // which 16-byte vector of a row
  const int row = lane / C::LPT;    // which of the TPI rows of a load

  unsigned char *stages = smem + warp * ST * C::STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::SMEM_STAGES) + warp * ST;
  float *mo = reinterpret_cast<float *>(smem + C::SMEM_STAGES + C::SMEM_BARS);  // [NW][G][D]
  float *mm = mo + NW * G * D;                                                   // [NW][G]
  float *ml = mm + NW * G;                                                       // [NW][G]
  int *abort_flag = reinterpret_cast<int *>(ml + NW * G);

  if (lane == 0) {
    for (int i = 0; i < ST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.seg_count)  // fixed partitions for the merge
    a.seg_count[static_cast<int64_t>(a.num_seqs) * a.num_q_heads] = 0;

  const uint64_t policy = l2_evict_first_policy();
  const int Hkv = a.num_kv_heads, B = a.num_seqs, PART = a.partition_size;
  const T *kc = static_cast<const T *>(a.k_cache);
  const T *vc = static_cast<const T *>(a.v_cache);

  uint32_t n_issued = 0, n_consumed = 0;  // ring counters (warp-uniform)
  uint32_t valid_bits = 0;                // lane 0: stage holds a real page
  int cur_s = 0, cur_base = 0;            // cursor: first partition index of sequence cur_s

  for (int item = blockIdx.x;; item += gridDim.x) {
    const int pw = item / Hkv;
    const int h = item - pw * Hkv;

    // ---- find the sequence that owns partition index pw (forward-only cursor)
    int ctx = -1;
    while (cur_s < B) {
      const int s = cur_s + lane;
      int P = 0, c = 0;
      if (s < B) {
        c = clamp_context(seq_context(a, s, err), a.ctx_cap, err);
        P = num_partitions(c, PART);
      }
      int incl = P;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, s < B && cur_base + incl > pw);
      if (hit) {
        const int L = __ffs(hit) - 1;
        cur_base += __shfl_sync(0xffffffffu, incl - P, L);
        ctx = __shfl_sync(0xffffffffu, c, L);
        cur_s += L;
        break;
      }
      cur_base += __shfl_sync(0xffffffffu, incl, 31);
      cur_s += 32;
    }
    if (ctx < 0) break;  // past the last item

    const int s = cur_s;
    const int p = pw - cur_base;
    const int P_s = num_partitions(ctx, PART);
    const int tok0 = p * PART;
    const int tok1 = min(tok0 + PART, ctx);
    const int pg0 = tok0 / kBlockSize;
    const int n_pages = tok1 > tok0 ? (tok1 - tok0 + kBlockSize - 1) / kBlockSize : 0;
    const int my_n = warp < n_pages ? (n_pages - warp + NW - 1) / NW : 0;
    const int32_t *bt_row = a.block_tables + seq_table_row(a, s) * a.max_blocks_per_seq;

    // ---- query group in registers, in base-2 score units
    float qf[G][C::E];
    {
      const T *qb = static_cast<const T *>(a.q) +
                    (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D + chunk * C::E;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        Unpack<Tag>::run(*reinterpret_cast<const uint4 *>(qb + g * D), qf[g]);
#pragma unroll
        for (int e = 0; e < C::E; ++e) qf[g][e] *= a.scale_log2;
      }
    }

    float m_run[G], l_run[G], acc[G][C::E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < C::E; ++e) acc[g][e] = 0.f;
    }

    // lane 0: start the copy of this warp's k-th page of the item into stage st
    auto issue = [&](int k, uint32_t st) {
      const int page = pg0 + warp + k * NW;
      const int blk = bt_row[page];
      if (blk >= 0 && blk < a.num_blocks) {
        const int64_t off = (static_cast<int64_t>(blk) * Hkv + h) * (kBlockSize * D);
        unsigned char *dst = stages + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES);
        bulk_copy_g2s(dst, kc + off, C::PAGE_BYTES, &bars[st], policy);
        bulk_copy_g2s(dst + C::PAGE_BYTES, vc + off, C::PAGE_BYTES, &bars[st], policy);
        valid_bits |= 1u << st;
      } else {
        atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
        mbar_arrive(&bars[st]);
        valid_bits &= ~(1u << st);
      }
    };

    const int pre = min(my_n, ST);
    if (lane == 0)
      for (int k = 0; k < pre; ++k) issue(k, (n_issued + k) % ST);
    n_issued += pre;

    bool timed_out = false;
    for (int k = 0; k < my_n; ++k) {
      const uint32_t st = n_consumed % ST;
      const uint32_t par = (n_consumed / ST) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], par, kWaitBudgetCycles));
      if (!ok) {
        if (lane == 0) atomicOr(err, PHOTON_DEVERR_WAIT_TIMEOUT);
        drain_async_copies();
        timed_out = true;
        break;
      }
      const bool valid = __shfl_sync(0xffffffffu, (valid_bits >> st) & 1u, 0) != 0;
      const int page_tok0 = (pg0 + warp + k * NW) * kBlockSize;
      const int nvalid = valid ? min(kBlockSize, tok1 - page_tok0) : 0;

      if (nvalid > 0) {
        const T *Ks = reinterpret_cast<const T *>(stages + st * C::STAGE_BYTES);
        const T *Vs = Ks + kBlockSize * D;
        float sc[C::ITERS][G];
        // scores: each lane dots its 16-byte slice of a row with the G queries
#pragma unroll
        for (int it = 0; it < C::ITERS; ++it) {
          float kf[C::E];
          Unpack<Tag>::run(
              *reinterpret_cast<const uint4 *>(Ks + (it * C::TPI + row) * D + chunk * C::E), kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float d0 = 0.f;
#pragma unroll
            for (int e = 0; e < C::E; ++e) d0 = fmaf(qf[g][e], kf[e], d0);
            sc[it][g] = d0;
          }
        }
        // finish the dot products across the LPT lanes of each row
#pragma unroll
        for (int it = 0; it < C::ITERS; ++it)
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int o = C::LPT / 2; o > 0; o >>= 1) sc[it][g] += warp_xor(sc[it][g], o);
        // rows past the context take no weight
#pragma unroll
        for (int it = 0; it < C::ITERS; ++it)
          if (it * C::TPI + row >= nvalid)
#pragma unroll
            for (int g = 0; g < G; ++g) sc[it][g] = -INFINITY;
        // online softmax update, per query head
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mx = sc[0][g];
#pragma unroll
          for (int it = 1; it < C::ITERS; ++it) mx = fmaxf(mx, sc[it][g]);
#pragma unroll
          for (int o = C::LPT; o < 32; o <<= 1) mx = fmaxf(mx, warp_xor(mx, o));
          const float m_new = fmaxf(m_run[g], mx);
          alpha[g] = exp2f(m_run[g] - m_new);
          m_run[g] = m_new;
          float ls = 0.f;
#pragma unroll
          for (int it = 0; it < C::ITERS; ++it) {
            const float pe = exp2f(sc[it][g] - m_new);
            sc[it][g] = pe;
            ls += pe;
          }
          l_run[g] = fmaf(l_run[g], alpha[g], ls);
#pragma unroll
          for (int e = 0; e < C::E; ++e) acc[g][e] *= alpha[g];
        }
        // weighted V rows
#pragma unroll
        for (int it = 0; it < C::ITERS; ++it) {
          float vf[C::E];
          Unpack<Tag>::run(
              *reinterpret_cast<const uint4 *>(Vs + (it * C::TPI + row) * D + chunk * C::E), vf);
          if (it * C::TPI + row >= nvalid)  // slots past the context may hold any bits
#pragma unroll
            for (int e = 0; e < C::E; ++e) vf[e] = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::E; ++e) acc[g][e] = fmaf(sc[it][g], vf[e], acc[g][e]);
        }
      }
      __syncwarp();
      ++n_consumed;
      if (k + ST < my_n) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(k + ST, st);
        }
        ++n_issued;
      }
    }
    // A timeout in any warp ends this CTA after the item.  The decision is
    // local to the CTA (the sticky error word only reports; a bit left set by
    // an earlier launch must not stop this one): other CTAs run on, each of
    // their waits is bounded too and each CTA gives up at most once, so the
    // launch still ends within about one wait budget per wave of CTAs.
    if (timed_out && lane == 0) *abort_flag = 1;

    // ---- combine the TPI row slots of each warp, then the NW warps
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = C::LPT; o < 32; o <<= 1) l_run[g] += warp_xor(l_run[g], o);
#pragma unroll
      for (int e = 0; e < C::E; ++e)
#pragma unroll
        for (int o = C::LPT; o < 32; o <<= 1) acc[g][e] += warp_xor(acc[g][e], o);
    }
    if (row == 0)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < C::E; ++e) mo[(warp * G + g) * D + chunk * C::E + e] = acc[g][e];
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mm[warp * G + g] = m_run[g];
        ml[warp * G + g] = l_run[g];
      }
    __syncthreads();
    if (*abort_flag) return;  // every thread sees the same flag after the barrier

    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
      const int g = idx / D, e = idx - (idx / D) * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * G + g]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = mm[w * G + g];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L = fmaf(ml[w * G + g], f, L);
        O = fmaf(mo[(w * G + g) * D + e], f, O);
      }
      const int64_t qrow = static_cast<int64_t>(s) * a.num_q_heads + h * G + g;
      if (P_s == 1) {
        const float r = L > 0.f ? O / L : 0.f;
        if (a.out_bf16)
          static_cast<__nv_bfloat16 *>(a.out)[qrow * D + e] = __float2bfloat16_rn(r);
        else
          static_cast<float *>(a.out)[qrow * D + e] = r;
      } else {
        const int64_t prow = qrow * a.max_partitions + p;
        a.o_part[prow * D + e] = O;
        if (e == 0) {
          a.m_part[prow] = M;
          a.l_part[prow] = L;
        }
      }
    }
    __syncthreads();
  }
}

// Merge of the partition partials of one (sequence, query head) per CTA:
// M = max_p m_p, L = sum_p l_p 2^(m_p - M), out = sum_p o_p 2^(m_p - M) / L.
// The maximum is taken by all threads over strided p and reduced in shared
// memory; then PG groups of D/4 threads split the partitions (group j takes
// p = j, j + PG, ...; each thread one float4 of the output), and the groups
// are summed through shared memory in a fixed order (deterministic).  Rows
// with a single partition were written by the partial kernel and are left
// alone.
template <int D>
struct ReduceCfg {
  static constexpr int TPR = D / 4;               // threads per partition group
  static constexpr int PG = D >= 256 ? 4 : 8;     // partition groups
  static constexpr int THREADS = TPR * PG;
};

template <int D>
__global__ void __launch_bounds__(ReduceCfg<D>::THREADS) lse_reduce_kernel(const DecodeArgs a) {
  using R = ReduceCfg<D>;
  __shared__ float4 s_o[R::PG][R::TPR];
  __shared__ float s_l[R::PG];
  __shared__ float s_m[R::THREADS / 32];
  pdl_launch_dependents();
  pdl_wait();
  const int64_t row = blockIdx.x;  // (sequence, query head)
  const int pg = threadIdx.x / R::TPR;
  const int x = threadIdx.x % R::TPR;
  const int s = static_cast<int>(row / a.num_q_heads);
  int P;
  if (a.seg_count && a.seg_count[static_cast<int64_t>(a.num_seqs) * a.num_q_heads] == 1) {
    // decode, page-balanced pieces: the count the partial kernel recorded for
    // this row (bounded by the row's slots whatever the word holds)
    P = min(a.seg_count[row], a.max_partitions);
  } else {
    // fixed partitions of the context (prefill: a token whose sequence row is
    // out of range has context 0; the partial kernels wrote its zero row)
    int ctx = !a.query_positions ? a.context_lens[s]
              : (a.row_of_seq[s] < 0 || a.row_of_seq[s] >= a.num_table_rows) ? 0
                                                                             : a.query_positions[s] + 1;
    ctx = ctx < 0 ? 0 : (ctx > a.ctx_cap ? a.ctx_cap : ctx);
    P = num_partitions(ctx, a.partition_size);
  }
  if (P <= 1) return;  // uniform over the CTA
  const float *mp = a.m_part + row * a.max_partitions;
  const float *lp = a.l_part + row * a.max_partitions;
  const float4 *op = reinterpret_cast<const float4 *>(a.o_part + row * a.max_partitions * D) + x;
  float M = -INFINITY;
  for (int p = threadIdx.x; p < P; p += R::THREADS) M = fmaxf(M, mp[p]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, warp_xor(M, o));
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < R::THREADS / 32; ++w) M = fmaxf(M, s_m[w]);
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
  for (int p = pg; p < P; p += R::PG) {
    const float mw = mp[p];
    const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
    L = fmaf(lp[p], f, L);
    const float4 v = op[p * (D / 4)];
    o.x = fmaf(v.x, f, o.x);
    o.y = fmaf(v.y, f, o.y);
    o.z = fmaf(v.z, f, o.z);
    o.w = fmaf(v.w, f, o.w);
  }
  s_o[pg][x] = o;
  if (x == 0) s_l[pg] = L;
  __syncthreads();
  if (pg != 0) return;
  L = 0.f;
  o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < R::PG; ++j) {
    L += s_l[j];
    o.x += s_o[j][x].x;
    o.y += s_o[j][x].y;
    o.z += s_o[j][x].z;
    o.w += s_o[j][x].w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  if (a.out_bf16) {
    uint2 w;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * inv, o.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z * inv, o.w * inv);
    w.x = *reinterpret_cast<const uint32_t *>(&lo);
    w.y = *reinterpret_cast<const uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.out) + row * D)[x] = w;
  } else {
    reinterpret_cast<float4 *>(static_cast<float *>(a.out) + row * D)[x] =
        make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  }
}

// Stage-ring depth: about 24 KiB of pages in flight per warp.
template <typename Tag, int D>
constexpr int decode_stages() {
  constexpr int stage = 2 * kBlockSize * D * Tag::kBytes;
  constexpr int st = (24 * 1024) / stage;
  return st < 2 ? 2 : (st > 8 ? 8 : st);
}

constexpr int kDecodeWarps = 4;

template <typename Tag, int D, int G>
cudaError_t launch_partial(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  constexpr int ST = decode_stages<Tag, D>();
  using C = DecodeCfg<Tag, D, G, kDecodeWarps, ST>;
  auto kern = paged_decode_partial_kernel<Tag, D, G, kDecodeWarps, ST>;
  static std::atomic<int> occupancy[64];  // resident CTAs per SM, per device (0 = not yet set up)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (occupancy[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecodeWarps * 32, C::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    occupancy[dev].store(occ > 0 ? occ : 1, std::memory_order_relaxed);
  }
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) *
                      occupancy[dev].load(std::memory_order_relaxed);
  const int grid = static_cast<int>(items < cap ? items : cap);
  if (grid == 0) return cudaSuccess;
  // persistent grid in the fixed item order: launched without programmatic
  // serialisation (see launch_mma_kern)
  kern<<<grid, kDecodeWarps * 32, C::SMEM_TOTAL, stream>>>(a, err);
  return cudaGetLastError();
}

template <typename Tag, int D>
cudaError_t dispatch_group(const DecodeArgs &a, unsigned int *err, cudaStream_t stream) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_partial<Tag, D, 1>(a, err, stream);
    case 2: return launch_partial<Tag, D, 2>(a, err, stream);
    case 4: return launch_partial<Tag, D, 4>(a, err, stream);
    case 8: return launch_partial<Tag, D, 8>(a, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
