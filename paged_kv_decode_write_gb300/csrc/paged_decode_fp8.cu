// Split-K paged decode attention over an FP8 (E4M3) KV cache with per-KV-head
// scales, head_dim 64 or 128, on the tensor cores.
//
// Same page pipeline, online softmax and partial/merge contract as the bf16
// tensor-core kernel (paged_decode_mma.cuh).  What differs:
//  * with a workspace the split-K work is page-balanced pieces (equal runs of
//    the page stream per group of H_kv warps, see the walker there) instead
//    of fixed partitions: the kernel issues ~235 instructions per 2 KiB page,
//    so fewer, longer pieces (no per-item q loads, conversions and epilogues
//    between them) and even loads per warp pay here;
//  * pages are half the bytes: per (block, KV head) K is [16 tokens][d] and V
//    is [d dims][16 tokens] (dims outer), each 16*d bytes, each fetched with
//    one bulk copy on the TMA engine;
//  * E4M3 values convert exactly to f16 in hardware (cvt.rn.f16x2.e4m3x2), so
//    the MMAs are f16 (q converted once per item), fp32 accumulation; the K
//    scale is folded into the score scale and the V scale into the output;
//  * P enters P V as one f16 operand (11 significant bits, relative error
//    <= 2^-12 per probability, far below the 4 bits of the E4M3 values it
//    weights), not as the high + remainder pair of the bf16 kernel, whose
//    8-bit bf16 P needs the second MMA;
//  * inside a page the tokens are visited in the order
//    logical 8nt + 2c + j -> physical row 4c + 2nt + j, the same for the
//    score fragments and the P V operand, so a lane's four tokens of a V
//    fragment are four consecutive bytes of one dim row: one 32-bit load,
//    two conversions, no byte permutes; K fragment loads are 16-byte chunks
//    (d 64: pairs of rows share a 128-byte line, bank-conflict free; d 128:
//    two chunks per row, two rows per quarter-warp on the same banks).
#include <atomic>
#include <type_traits>
#include <cuda_fp16.h>

#include "paged_decode.cuh"
#include "paged_decode_mma.cuh"

namespace photon {
namespace {

template <int D>
struct Fp8Cfg {
  static_assert(D == 64 || D == 128, "FP8 decode: head_dim 64 or 128");
  static constexpr int PAGE = kBlockSize * D;  // bytes of K (or V) of one page
  static constexpr int PAIR = 2 * PAGE;        // K + V of one page
  static constexpr int KT = D / 16;            // k-steps of Q K^T
  static constexpr int KW = D / 8;             // f16x2 words of a K row per thread
  static constexpr int KCH = D / 64;           // 16-byte E4M3 chunks of a K row per thread
  static constexpr int MT = D / 16;            // m-tiles (16 dims) of V^T P^T
};

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 codes of a 32-bit word -> two f16x2 words (exact), splitting the
// word into its 16-bit halves inside PTX (no separate extract instructions).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t raw, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(raw));
}

constexpr int kFp8PagesPerStage = 2;  // one pipeline step covers 32 tokens

template <int D, int G, int NW, int ST, bool BAL>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_fp8_kernel(const DecodeArgs a, const float *__restrict__ k_scale,
                            const float *__restrict__ v_scale, unsigned int *err) {
  using C = Fp8Cfg<D>;
  constexpr int PP = kFp8PagesPerStage;
  constexpr int kFp8Page = C::PAGE;
  constexpr int kFp8Stage = C::PAIR;
  constexpr int STAGE = PP * kFp8Stage;  // [K page 0][K page 1][V page 0][V page 1]
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  unsigned char *stages = smem + warp * ST * STAGE;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * ST * STAGE) + warp * ST;
  const uint32_t stages_s = smem_addr(stages);
  if (lane == 0) {
    for (int i = 0; i < ST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if constexpr (BAL) prefetch_tables_l2(a);
  pdl_launch_dependents();

  const uint64_t policy = l2_evict_first_policy();
  const int total_warps = gridDim.x * NW;
  const unsigned char *kc = static_cast<const unsigned char *>(a.k_cache);
  const unsigned char *vc = static_cast<const unsigned char *>(a.v_cache);

  // K rows of this lane's n-tiles (column g) within a page; the lane's head
  // dims are D/4 consecutive ones, 16-byte chunks KCH*c .. KCH*c + KCH - 1
  uint32_t koff[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) koff[nt] = (4 * (g >> 1) + 2 * nt + (g & 1)) * D + 16 * C::KCH * c;
  // V dim rows 16mt + g (and +8), bytes 4c..4c+3 = tokens 4c..4c+3 of the page
  const uint32_t voff = PP * kFp8Page + g * 16 + 4 * c;

  Walker prod, cons;
  walker_start<BAL>(prod, a, lane, err, blockIdx.x * NW + warp, total_warps);
  walker_start<BAL>(cons, a, lane, err, blockIdx.x * NW + warp, total_warps);
  // the above reads only the batch's metadata: under programmatic launch it
  // runs beside the preceding kernel; pages, q and the workspace wait for it
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.seg_count)  // the merge's mode
    a.seg_count[static_cast<int64_t>(a.num_seqs) * a.num_q_heads] = BAL ? 1 : 0;
  uint32_t n_issued = 0, valid_bits = 0;  // lane 0: 2 bits per stage
  uint32_t c_slot = 0, c_phase = 0;      // consumer's ring slot and its phase parity
  int bt_base = INT_MIN / 2, bt_reg = -1;

  // Issues the producer's next pair of pages (the second may be past the item).
  auto issue_next = [&]() -> bool {
    while (prod.valid && prod.page >= prod.n_pages) {
      walker_next<BAL>(prod, a, lane, err, total_warps);
      bt_base = INT_MIN / 2;
    }
    if (!prod.valid) return false;
    if (prod.page + 1 - bt_base >= 32) {
      bt_base = prod.page;
      bt_reg = bt_base + lane < prod.n_pages
                   ? a.block_tables[seq_table_row(a, prod.s) * a.max_blocks_per_seq +
                                    prod.pg0 + bt_base + lane]
                   : -1;
    }
    const int blk0 = __shfl_sync(0xffffffffu, bt_reg, prod.page - bt_base);
    const int blk1 = __shfl_sync(0xffffffffu, bt_reg, prod.page + 1 - bt_base);
    const bool has1 = prod.page + 1 < prod.n_pages;
    const uint32_t st = n_issued % ST;
    if (lane == 0) {
      const bool ok0 = blk0 >= 0 && blk0 < a.num_blocks;
      const bool ok1 = has1 && blk1 >= 0 && blk1 < a.num_blocks;
      if (!ok0 || (has1 && !ok1)) atomicOr(err, PHOTON_DEVERR_BLOCK_RANGE);
      unsigned char *dst = stages + st * STAGE;
      const uint32_t bytes = (ok0 ? kFp8Stage : 0) + (ok1 ? kFp8Stage : 0);
      fence_proxy_async_smem();
      if (bytes) {
        mbar_arrive_expect_tx(&bars[st], bytes);
        if (ok0) {
          const int64_t off = (static_cast<int64_t>(blk0) * a.num_kv_heads + prod.h) * kFp8Page;
          bulk_copy_g2s(dst, kc + off, kFp8Page, &bars[st], policy);
          bulk_copy_g2s(dst + PP * kFp8Page, vc + off, kFp8Page, &bars[st], policy);
        }
        if (ok1) {
          const int64_t off = (static_cast<int64_t>(blk1) * a.num_kv_heads + prod.h) * kFp8Page;
          bulk_copy_g2s(dst + kFp8Page, kc + off, kFp8Page, &bars[st], policy);
          bulk_copy_g2s(dst + PP * kFp8Page + kFp8Page, vc + off, kFp8Page, &bars[st], policy);
        }
      } else {
        mbar_arrive(&bars[st]);
      }
      valid_bits = (valid_bits & ~(3u << (2 * st))) | ((ok0 ? 1u : 0u) << (2 * st)) |
                   ((ok1 ? 1u : 0u) << (2 * st + 1));
    }
    prod.page += PP;
    ++n_issued;
    return true;
  };
  for (int k = 0; k < ST; ++k)
    if (!issue_next()) break;

  uint32_t qa[C::KT][2];
  float o[C::MT][4];
  float m_run = -INFINITY, l_run = 0.f, sk = 0.f, vsc = 0.f;

  while (cons.valid) {
    if (cons.page == 0) {
      uint32_t qw[C::KW];
      if (g < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const __nv_bfloat16 *>(a.q) +
            (static_cast<int64_t>(cons.s) * a.num_q_heads + cons.h * G + g) * D + (D / 4) * c);
#pragma unroll
        for (int i = 0; i < C::KW / 4; ++i) {
          const uint4 v = src[i];
          qw[4 * i] = bf16x2_to_f16x2(v.x);
          qw[4 * i + 1] = bf16x2_to_f16x2(v.y);
          qw[4 * i + 2] = bf16x2_to_f16x2(v.z);
          qw[4 * i + 3] = bf16x2_to_f16x2(v.w);
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
      sk = a.scale_log2 * k_scale[cons.h];
      vsc = v_scale[cons.h];
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
      const uint32_t vb = __shfl_sync(0xffffffffu, (valid_bits >> (2 * st)) & 3u, 0);
      int nvalid[PP];
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        const int page_tok0 = (cons.pg0 + cons.page + pp) * kBlockSize;
        nvalid[pp] = ((vb >> pp) & 1u) ? max(0, min(kBlockSize, cons.tok1 - page_tok0)) : 0;
      }
      const uint32_t base = stages_s + st * STAGE;
      if (nvalid[0] + nvalid[1] > 0) {  // both pages skipped (bad block ids): nothing to add
      // ---- S^T for both pages: n-tiles 2pp + nt
      float s[PP][2][4];
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t raw[4 * C::KCH];
#pragma unroll
          for (int ch = 0; ch < C::KCH; ++ch)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(raw[4 * ch]), "=r"(raw[4 * ch + 1]), "=r"(raw[4 * ch + 2]),
                           "=r"(raw[4 * ch + 3])
                         : "r"(base + pp * kFp8Page + koff[nt] + 16 * ch));
          uint32_t kw[C::KW];
#pragma unroll
          for (int i = 0; i < 4 * C::KCH; ++i) e4m3x4_to_f16(raw[i], kw[2 * i], kw[2 * i + 1]);
          s[pp][nt][0] = s[pp][nt][1] = s[pp][nt][2] = s[pp][nt][3] = 0.f;
#pragma unroll
          for (int kt = 0; kt < C::KT; ++kt)
            mma_f16_16816(s[pp][nt], qa[kt][0], 0u, qa[kt][1], 0u, kw[2 * kt], kw[2 * kt + 1]);
        }
      // score (pp, nt, j) of head g is physical row 4c + 2nt + j of page pp
      float mx = -INFINITY;
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) s[pp][nt][j] *= sk;
      if (nvalid[0] + nvalid[1] < PP * kBlockSize) {  // a partial page: mask its tail
#pragma unroll
        for (int pp = 0; pp < PP; ++pp)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (4 * c + 2 * nt + j >= nvalid[pp]) s[pp][nt][j] = -INFINITY;
      }
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mx = fmaxf(mx, fmaxf(s[pp][nt][0], s[pp][nt][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);  // finite: the first page always has tokens
      const float alpha = exp2_approx(m_run - m_new);
      m_run = m_new;
      float ps = 0.f;
      uint32_t ph[PP][2];
#pragma unroll
      for (int pp = 0; pp < PP; ++pp)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float p0 = exp2_approx(s[pp][nt][0] - m_new);
          const float p1 = exp2_approx(s[pp][nt][1] - m_new);
          ps += p0 + p1;
          ph[pp][nt] = pack_f16(p0, p1);
        }
      l_run = fmaf(l_run, alpha, ps);
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * c);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      // ---- O^T += V^T P^T, page by page
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        // tokens 4c.. past the context: zero (their bytes may hold anything);
        // full pages (the rule) skip the masking
        auto pv_page = [&](auto masked_tag) {
          constexpr bool masked = decltype(masked_tag)::value;
          uint32_t vmask = 0xffffffffu;
          if (masked) {
            const int nv = min(max(nvalid[pp] - 4 * c, 0), 4);
            vmask = nv >= 4 ? 0xffffffffu : ((1u << (8 * nv)) - 1u);
          }
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            uint32_t w0, w1;
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=r"(w0)
                         : "r"(base + pp * kFp8Page + voff + mt * 256));
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=r"(w1)
                         : "r"(base + pp * kFp8Page + voff + mt * 256 + 128));
            if (masked) {
              w0 &= vmask;
              w1 &= vmask;
            }
            uint32_t va0, va1, va2, va3;
            e4m3x4_to_f16(w0, va0, va2);  // dim 16mt+g: tokens (2c, 2c+1) and (8+2c, 9+2c)
            e4m3x4_to_f16(w1, va1, va3);  // dim 16mt+8+g
            mma_f16_16816(o[mt], va0, va1, va2, va3, ph[pp][0], ph[pp][1]);
          }
        };
        if (nvalid[pp] < kBlockSize)
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
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const float l0 = __shfl_sync(0xffffffffu, l, 8 * c);
      const float l1 = __shfl_sync(0xffffffffu, l, 8 * c + 4);
      const float m0 = __shfl_sync(0xffffffffu, m_run, 8 * c);
      const float m1 = __shfl_sync(0xffffffffu, m_run, 8 * c + 4);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int head = 2 * c + j;
        if (head >= G) continue;
        const float lj = j ? l1 : l0;
        const int64_t qrow = static_cast<int64_t>(cons.s) * a.num_q_heads + cons.h * G + head;
        if constexpr (BAL)
          if (g == 0 && cons.p == 0) a.seg_count[qrow] = cons.P_s;
        if (cons.P_s == 1) {
          const float f = lj > 0.f ? vsc / lj : 0.f;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int64_t idx = qrow * D + 16 * mt + 8 * r + g;
              const float val = o[mt][2 * r + j] * f;
              if (a.out_bf16)
                static_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(val);
              else
                static_cast<float *>(a.out)[idx] = val;
            }
        } else {
          const int64_t prow = qrow * a.max_partitions + cons.p;
          float *dst = a.o_part + prow * D;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) dst[16 * mt + 8 * r + g] = o[mt][2 * r + j] * vsc;
          if (g == 0) {
            a.m_part[prow] = j ? m1 : m0;
            a.l_part[prow] = lj;
          }
        }
      }
      walker_next<BAL>(cons, a, lane, err, total_warps);
    }
  }
}

// Ring depth: 2 two-page stages (8 KiB per warp at d 64: registers, not
// shared memory, then bound occupancy at 5 CTAs of 4 warps per SM; same-box
// 3 -> 2 stages: long-context step 0.834 -> 0.781 ms; 16 KiB per warp at
// d 128, 3 CTAs per SM).
template <int D, int G, bool BAL>
cudaError_t launch_fp8_kern(const DecodeArgs &a, const float *k_scale, const float *v_scale,
                            unsigned int *err, cudaStream_t stream) {
  constexpr int NW = 4, ST = 2;
  constexpr int SMEM = NW * ST * kFp8PagesPerStage * Fp8Cfg<D>::PAIR + NW * ST * 8;
  auto kern = paged_decode_fp8_kernel<D, G, NW, ST, BAL>;
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
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.max_partitions * a.num_kv_heads;
  const int64_t warps_cap = static_cast<int64_t>(device_sm_count()) *
                            occupancy[dev].load(std::memory_order_relaxed) * NW;
  const int64_t warps = items < warps_cap ? items : warps_cap;
  const int grid = static_cast<int>((warps + NW - 1) / NW);
  if (grid == 0) return cudaSuccess;
  DecodeArgs la = a;
  la.balanced = BAL ? 1 : 0;
  // Programmatic launch: the CTAs start behind the preceding kernel (the
  // step's small write) and run the metadata prologue before
  // griddepcontrol.wait.  Same GPU, full grids: Qwen3 batch-64 step 71.9 ->
  // 67.1 us, long-context step 0.676 -> 0.671 ms (kernel alone unchanged).
  return launch_pdl(kern, dim3(grid), dim3(NW * 32), SMEM, stream, la, k_scale, v_scale, err);
}

template <int D, int G>
cudaError_t launch_fp8(const DecodeArgs &a, const float *k_scale, const float *v_scale,
                       unsigned int *err, cudaStream_t stream) {
  if (balanced_pieces(a)) return launch_fp8_kern<D, G, true>(a, k_scale, v_scale, err, stream);
  return launch_fp8_kern<D, G, false>(a, k_scale, v_scale, err, stream);
}

}  // namespace

template <int D>
cudaError_t dispatch_fp8_group(const DecodeArgs &a, const float *k_scale, const float *v_scale,
                               unsigned int *err, cudaStream_t st) {
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_fp8<D, 1>(a, k_scale, v_scale, err, st);
    case 2: return launch_fp8<D, 2>(a, k_scale, v_scale, err, st);
    case 4: return launch_fp8<D, 4>(a, k_scale, v_scale, err, st);
    case 8: return launch_fp8<D, 8>(a, k_scale, v_scale, err, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_partial_fp8(const DecodeArgs &a, const float *k_scale,
                                      const float *v_scale, unsigned int *err, cudaStream_t st) {
  switch (a.head_dim) {
    case 64: return dispatch_fp8_group<64>(a, k_scale, v_scale, err, st);
    case 128: return dispatch_fp8_group<128>(a, k_scale, v_scale, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
