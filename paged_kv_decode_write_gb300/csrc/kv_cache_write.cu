// Batched KV-cache write with fused RoPE (sm_103a).
//
// PhotonInfer README, "Technical details > Paged attention": one kernel
// writes K/V for many sequences; "Key features > GPU-optimised kernels":
// batched RoPE as a fused operation.
//
// One CTA per written token, and a short dependency chain per CTA: the
// token's K and V rows are copied to shared memory asynchronously (cp.async)
// first; while they are in flight the threads compute the position's
// rotation table -- the fp64 sine and cosine of pos * theta^(-2i/d), the
// angle reduced to [-pi, pi] -- then one barrier, V stored as 16-byte bit
// copies and K rotated.  A rotated element is the storage type's nearest
// value to the exact x*cos - y*sin (one unit in the last place at worst,
// whatever the cancellation): computed in fp32 with an error bound and kept
// when the bound cannot change the rounding, recomputed from fp64 products
// when it could (bf16; rare).  fp32 caches rotate in fp64 throughout.  The
// FP8 write takes the same route to its E4M3 codes.  The loops stay rolled:
// each SM runs one or two of these CTAs once, so the instruction stream is
// fetched cold and the kernel's code size shows in its time.
#include "common.cuh"
#include "internal.h"

namespace photon {
namespace {

// 2*pi = kTwoPiHi + kTwoPiLo: kTwoPiHi holds the leading 30 significant bits
// (so k * kTwoPiHi is exact for |k| < 2^23) and kTwoPiLo the remainder,
// rounded to double.  Used to reduce angles before sincos.
constexpr double kTwoPiHi = 0x1.921fb548p+2;
constexpr double kTwoPiLo = -0x1.de973dcb3b39ap-29;
constexpr double kInvTwoPi = 0x1.45f306dc9c883p-3;

// Nearest-even bf16 of a double in one rounding: truncate to float, keep an
// inexact-sticky bit in the last place (round-to-odd), then round the float
// to bf16.  Round-to-odd to 24 bits followed by round-to-nearest to 8 bits
// equals direct rounding to 8 bits (Boldo & Melquiond, "Emulation of FMA and
// correctly rounded sums: proved algorithms using rounding to odd", 2008).
__device__ __forceinline__ __nv_bfloat16 f64_to_bf16(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  return __float2bfloat16_rn(f);
}

constexpr int kWriteThreads = 64;
constexpr int kStageBytes = 8192;  // K and V rows of one round, staged in shared memory

// Query heads one CTA rotates: as many as its threads cover pair by pair.
__host__ __device__ __forceinline__ int q_heads_per_cta(int head_dim) {
  const int h = kWriteThreads / (head_dim / 2);
  return h > 0 ? h : 1;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Starts the copy of `bytes` (a multiple of 16) from src to shared memory.
__device__ __forceinline__ void stage_async(unsigned char *dst, const void *src, int bytes) {
  for (int o = 16 * static_cast<int>(threadIdx.x); o < bytes; o += 16 * kWriteThreads)
    cp_async16(dst + o, static_cast<const unsigned char *>(src) + o);
}

// Rotation table of one position: cs[i] = (cos, sin) of pos * inv_freq[i] in
// fp64 (the angle first reduced to [-pi, pi] with the two-term 2*pi), cs32
// the same rounded to fp32.  Visible after the caller's next barrier.
__device__ __forceinline__ void rope_table(const WriteArgs &a, int pos, double (*cs)[2],
                                           float (*cs32)[2]) {
  const double p = static_cast<double>(pos);
#pragma unroll 1
  for (int i = threadIdx.x; i < a.head_dim / 2; i += kWriteThreads) {
    const double ang = p * a.inv_freq[i];
    const double k = rint(ang * kInvTwoPi);
    double sn, c;
    sincos(fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, ang)), &sn, &c);
    cs[i][0] = c;
    cs[i][1] = sn;
    cs32[i][0] = static_cast<float>(c);
    cs32[i][1] = static_cast<float>(sn);
  }
}

// The rare fp64 decisions, out of line (kept off the instruction stream of
// the common path).
__device__ __noinline__ __nv_bfloat16 rotate_bf16_fp64(float u, float w, double c, double t) {
  return f64_to_bf16(static_cast<double>(u) * c + static_cast<double>(w) * t);
}

// One rotated element y = u*c + w*t (t = -sin for the first of a pair, +sin
// for the second) of pair i, rounded once from its exact value into the
// storage type.
template <typename Tag>
struct Rotate;

template <>
struct Rotate<F32Tag> {
  // fp64 products, one rounding to fp32
  __device__ __forceinline__ static float run(float u, float w, float, float, const double (*cs)[2],
                                              int i, bool first) {
    const double t = first ? -cs[i][1] : cs[i][1];
    return __double2float_rn(static_cast<double>(u) * cs[i][0] + static_cast<double>(w) * t);
  }
};

template <>
struct Rotate<BF16Tag> {
  // fp32 first: y = fl(u*c32 + fl(w*t32)) with c32, t32 the fp32 roundings of
  // the fp64 cos / sin is within 2^-23 * (|u| + |w| + |y|) of the exact
  // u*c + w*t (three relative roundings of 2^-24, |cos|, |sin| <= 1).  With
  // twice that margin, if y - e and y + e round to the same bf16, so does
  // the exact value (rounding is monotonic), and that bf16 is the answer.
  // Otherwise -- a value within the margin of a rounding boundary, rare --
  // the fp64 products decide.
  __device__ __forceinline__ static __nv_bfloat16 run(float u, float w, float c32, float t32,
                                                      const double (*cs)[2], int i, bool first) {
    const float y = fmaf(u, c32, w * t32);
    const float e = fmaf(fabsf(y) + fabsf(u) + fabsf(w), 0x1p-22f, 0x1p-126f);
    const __nv_bfloat16 lo = __float2bfloat16_rn(y - e);
    const __nv_bfloat16 hi = __float2bfloat16_rn(y + e);
    if (__bfloat16_as_ushort(lo) == __bfloat16_as_ushort(hi)) return lo;
    return rotate_bf16_fp64(u, w, cs[i][0], first ? -cs[i][1] : cs[i][1]);
  }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Rotates nrows staged rows (shared memory, [nrows][d]) into dst (row r at
// dst + r * dst_stride), pair by pair.
template <typename Tag>
__device__ __forceinline__ void rotate_rows(const WriteArgs &a, const typename Tag::T *src,
                                            typename Tag::T *dst, int64_t dst_stride, int nrows,
                                            const double (*cs)[2], const float (*cs32)[2]) {
  const int D = a.head_dim, half = D / 2;
  const bool gptj = a.rope_style == PHOTON_ROPE_GPTJ;
  for (int idx = threadIdx.x; idx < nrows * half; idx += kWriteThreads) {
    const int r = idx / half, i = idx - r * half;
    const int e0 = gptj ? 2 * i : i, e1 = gptj ? 2 * i + 1 : i + half;
    const float x0 = to_f32(src[r * D + e0]), x1 = to_f32(src[r * D + e1]);
    const float c32 = cs32[i][0], s32 = cs32[i][1];
    typename Tag::T *row = dst + r * dst_stride;
    row[e0] = Rotate<Tag>::run(x0, x1, c32, -s32, cs, i, true);
    row[e1] = Rotate<Tag>::run(x1, x0, c32, s32, cs, i, false);
  }
}

// Copies nrows staged rows (shared memory, [nrows][d]) to dst (row r at
// dst + r * dst_stride) in 16-byte chunks.
template <typename Tag>
__device__ __forceinline__ void store_rows(const typename Tag::T *src, typename Tag::T *dst,
                                           int64_t dst_stride, int nrows, int D) {
  constexpr int E = 16 / sizeof(typename Tag::T);
  const int per_row = D / E;
  for (int idx = threadIdx.x; idx < nrows * per_row; idx += kWriteThreads) {
    const int r = idx / per_row, ch = idx - r * per_row;
    reinterpret_cast<uint4 *>(dst + r * dst_stride)[ch] =
        reinterpret_cast<const uint4 *>(src + r * D)[ch];
  }
}

// Rotates heads [h0, h0 + q_heads_per_cta) of query row `row`
// ([num_q_heads][head_dim]) in place at q_positions[row].
template <typename Tag>
__device__ __forceinline__ void rotate_q_part(const WriteArgs &a, int row, int h0,
                                              unsigned char *stage, double (*cs)[2],
                                              float (*cs32)[2]) {
  using T = typename Tag::T;
  if (a.rope_style == PHOTON_ROPE_NONE) return;
  const int D = a.head_dim;
  const int nrows = min(a.num_q_heads, h0 + q_heads_per_cta(D)) - h0;
  T *q = static_cast<T *>(a.q) + (static_cast<int64_t>(row) * a.num_q_heads + h0) * D;
  stage_async(stage, q, nrows * D * static_cast<int>(sizeof(T)));  // <= 64 pairs (or one d-256 head)
  rope_table(a, a.q_positions[row], cs, cs32);
  cp_async_wait_all();
  __syncthreads();
  rotate_rows<Tag>(a, reinterpret_cast<const T *>(stage), q, D, nrows, cs, cs32);
}

// One CTA per written token (and, when q is given, per group of query heads
// of a query row).  Per round of KV heads: the token's K and V rows are
// copied to shared memory asynchronously while the threads compute the
// position's rotation table (first round), then V rows are stored as they
// are and K rows rotated.
template <typename Tag>
__global__ void __launch_bounds__(kWriteThreads)
    kv_cache_write_kernel(const __grid_constant__ WriteArgs a, unsigned int *err) {
  using T = typename Tag::T;
  __shared__ __align__(16) unsigned char stage[kStageBytes];
  __shared__ double cs[kMaxRopePairs][2];
  __shared__ float cs32[kMaxRopePairs][2];
  pdl_wait();
  pdl_launch_dependents();  // after the wait: a dependent decode grid meets only this small one
  if (static_cast<int>(blockIdx.x) >= a.num_tokens) {  // part of a query row: rotate in place
    const int hpc = q_heads_per_cta(a.head_dim);
    const int per_row = (a.num_q_heads + hpc - 1) / hpc;
    const int qb = blockIdx.x - a.num_tokens;
    rotate_q_part<Tag>(a, qb / per_row, (qb % per_row) * hpc, stage, cs, cs32);
    return;
  }
  const int64_t t = blockIdx.x;
  const int D = a.head_dim, H = a.num_kv_heads;
  const int row_bytes = D * static_cast<int>(sizeof(T));
  const int rpc = max(1, kStageBytes / (2 * row_bytes));  // KV heads per round
  const bool rotate = a.rope_style != PHOTON_ROPE_NONE;
  const T *k = static_cast<const T *>(a.k) + t * H * D;
  const T *v = static_cast<const T *>(a.v) + t * H * D;
  T *sk = reinterpret_cast<T *>(stage);
  T *sv = reinterpret_cast<T *>(stage + kStageBytes / 2);
  int n = min(H, rpc);
  stage_async(stage, k, n * row_bytes);
  stage_async(stage + kStageBytes / 2, v, n * row_bytes);
  const int64_t slot = a.slot_mapping[t];
  if (rotate) rope_table(a, a.positions[t], cs, cs32);
  if (slot < 0 || slot >= a.num_slots) {
    if (slot >= a.num_slots && threadIdx.x == 0) atomicOr(err, PHOTON_DEVERR_SLOT_RANGE);
    cp_async_wait_all();
    return;
  }
  const int64_t blk = slot / kBlockSize, off = slot - blk * kBlockSize;
  // head h of the token goes to cache row (blk * H + h) * block_size + off
  const int64_t dst_stride = static_cast<int64_t>(kBlockSize) * D;
  T *kd = static_cast<T *>(a.k_cache) + (blk * H * kBlockSize + off) * D;
  T *vd = static_cast<T *>(a.v_cache) + (blk * H * kBlockSize + off) * D;
  for (int h0 = 0;;) {
    cp_async_wait_all();
    __syncthreads();
    store_rows<Tag>(sv, vd + h0 * dst_stride, dst_stride, n, D);
    if (rotate)
      rotate_rows<Tag>(a, sk, kd + h0 * dst_stride, dst_stride, n, cs, cs32);
    else
      store_rows<Tag>(sk, kd + h0 * dst_stride, dst_stride, n, D);
    h0 += n;
    if (h0 >= H) break;
    n = min(H - h0, rpc);
    __syncthreads();  // the round's rows are read before the next round overwrites them
    stage_async(stage, k + h0 * D, n * row_bytes);
    stage_async(stage + kStageBytes / 2, v + h0 * D, n * row_bytes);
  }
}

// Nearest E4M3 of a double in one rounding, saturating at +-448: round-to-odd
// into float (24 bits), then the hardware's round-to-nearest-even conversion
// to E4M3 (4 significant bits) with saturation -- the same two-step argument
// as for bf16 above.
__device__ __forceinline__ unsigned char f64_to_e4m3(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(f));
  return static_cast<unsigned char>(r & 0xffu);
}

// Code of x / scale from the fp64 quotient (IEEE division, one rounding):
// for float x and scale it lies on the same side of every E4M3 rounding
// boundary as the exact quotient, and on an exact midpoint it is the
// midpoint itself, which the conversion sends to the even code.
__device__ __noinline__ unsigned char e4m3_fp64(double x, float scale) {
  return f64_to_e4m3(__ddiv_rn(x, static_cast<double>(scale)));
}

// Nearest E4M3 code (round to nearest even, saturating at +-448) of a real
// value known to lie within e of the fp32 value y: when y - e and y + e give
// the same code, every value between them does (rounding is monotonic) and
// that code is returned; otherwise returns -1.
__device__ __forceinline__ int e4m3_if_decided(float y, float e) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(y + e), "f"(y - e));
  return (r >> 8) == (r & 0xffu) ? static_cast<int>(r & 0xffu) : -1;
}

// FP8 cache write: K pool [blocks][H_kv][bs][d] and V pool [blocks][H_kv][d][bs]
// of E4M3 codes; code = round(x / scale[h]) of the exact value x (RoPE'd for
// K).  Decided in fp32 first: with is32 the fp32 reciprocal, y = fl(x * is32)
// is within 2^-23 (|x| |is32| + |y|) of the exact quotient (for K, x itself is
// the fp32 rotation, whose own margin adds 2^-23 (|u| + |w| + |x|) |is32|);
// with twice the margin the code is taken when both ends agree, from the fp64
// quotient otherwise (values near a rounding boundary of the 4-bit E4M3 grid,
// exact midpoints included: rare).  Rounds of KV heads are staged in shared
// memory as in kv_cache_write_kernel.
template <typename Tag>
__global__ void __launch_bounds__(kWriteThreads)
    kv_cache_write_fp8_kernel(const __grid_constant__ WriteArgs a, const float *k_scale,
                              const float *v_scale, unsigned int *err) {
  using T = typename Tag::T;
  __shared__ __align__(16) unsigned char stage[kStageBytes];
  __shared__ double cs[kMaxRopePairs][2];
  __shared__ float cs32[kMaxRopePairs][2];
  pdl_wait();
  pdl_launch_dependents();  // after the wait: a dependent decode grid meets only this small one
  const int64_t t = blockIdx.x;
  const int D = a.head_dim, half = D / 2, H = a.num_kv_heads;
  const int row_bytes = D * static_cast<int>(sizeof(T));
  const int rpc = max(1, kStageBytes / (2 * row_bytes));
  const bool rotate = a.rope_style != PHOTON_ROPE_NONE;
  const bool gptj = a.rope_style == PHOTON_ROPE_GPTJ;
  const T *k = static_cast<const T *>(a.k) + t * H * D;
  const T *v = static_cast<const T *>(a.v) + t * H * D;
  const T *sk = reinterpret_cast<const T *>(stage);
  const T *sv = reinterpret_cast<const T *>(stage + kStageBytes / 2);
  int n = min(H, rpc);
  stage_async(stage, k, n * row_bytes);
  stage_async(stage + kStageBytes / 2, v, n * row_bytes);
  const int64_t slot = a.slot_mapping[t];
  if (rotate) {
    rope_table(a, a.positions[t], cs, cs32);
  } else {
    for (int i = threadIdx.x; i < half; i += kWriteThreads) {
      cs[i][0] = 1.0, cs[i][1] = 0.0;
      cs32[i][0] = 1.f, cs32[i][1] = 0.f;
    }
  }
  if (slot < 0 || slot >= a.num_slots) {
    if (slot >= a.num_slots && threadIdx.x == 0) atomicOr(err, PHOTON_DEVERR_SLOT_RANGE);
    cp_async_wait_all();
    return;
  }
  const int64_t blk = slot / kBlockSize, off = slot - blk * kBlockSize;
  unsigned char *vc = static_cast<unsigned char *>(a.v_cache);
  unsigned char *kc = static_cast<unsigned char *>(a.k_cache);
  for (int h0 = 0;;) {
    cp_async_wait_all();
    __syncthreads();
    // V: element e of head h -> byte ((blk * H + h) * d + e) * bs + off
    for (int idx = threadIdx.x; idx < n * D; idx += kWriteThreads) {
      const int r = idx / D, e = idx - r * D, h = h0 + r;
      const float sc = v_scale[h];
      const float is = __frcp_rn(sc);
      const float x = to_f32(sv[idx]);
      const float y = x * is;
      int code = e4m3_if_decided(y, fmaf(fabsf(x) * fabsf(is) + fabsf(y), 0x1p-22f, 0x1p-126f));
      if (code < 0) code = e4m3_fp64(static_cast<double>(x), sc);
      vc[((blk * H + h) * D + e) * kBlockSize + off] = static_cast<unsigned char>(code);
    }
    // K: rotated pair (e0, e1) of head h -> bytes ((blk * H + h) * bs + off) * d + e
    for (int idx = threadIdx.x; idx < n * half; idx += kWriteThreads) {
      const int r = idx / half, i = idx - r * half, h = h0 + r;
      const int e0 = gptj ? 2 * i : i, e1 = gptj ? 2 * i + 1 : i + half;
      const float sc = k_scale[h];
      const float is = __frcp_rn(sc);
      unsigned char *row = kc + ((blk * H + h) * kBlockSize + off) * D;
      const float x0 = to_f32(sk[r * D + e0]), x1 = to_f32(sk[r * D + e1]);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const float u = m ? x1 : x0, w = m ? x0 : x1;
        const float tt32 = m ? cs32[i][1] : -cs32[i][1];
        const float rr = fmaf(u, cs32[i][0], w * tt32);
        const float y = rr * is;
        const float e = fmaf(fabsf(is) * (fabsf(u) + fabsf(w) + 2.f * fabsf(rr)) + fabsf(y),
                             0x1p-22f, 0x1p-126f);
        int code = e4m3_if_decided(y, e);
        if (code < 0)
          code = e4m3_fp64(static_cast<double>(u) * cs[i][0] +
                               static_cast<double>(w) * (m ? cs[i][1] : -cs[i][1]),
                           sc);
        row[m ? e1 : e0] = static_cast<unsigned char>(code);
      }
    }
    h0 += n;
    if (h0 >= H) break;
    n = min(H - h0, rpc);
    __syncthreads();
    stage_async(stage, k + h0 * D, n * row_bytes);
    stage_async(stage + kStageBytes / 2, v + h0 * D, n * row_bytes);
  }
}

}  // namespace

cudaError_t launch_kv_cache_write_fp8(const WriteArgs &a, photon_dtype in_dt, const float *k_scale,
                                      const float *v_scale, unsigned int *err, cudaStream_t st) {
  if (a.num_tokens == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.num_tokens));
  if (in_dt == PHOTON_BF16)
    return launch_pdl(kv_cache_write_fp8_kernel<BF16Tag>, grid, dim3(kWriteThreads), 0, st, a,
                      k_scale, v_scale, err);
  return launch_pdl(kv_cache_write_fp8_kernel<F32Tag>, grid, dim3(kWriteThreads), 0, st, a,
                    k_scale, v_scale, err);
}

cudaError_t launch_kv_cache_write(const WriteArgs &a, photon_dtype dt, unsigned int *err,
                                  cudaStream_t st) {
  const int hpc = q_heads_per_cta(a.head_dim);
  const int64_t q_blocks =
      a.q ? static_cast<int64_t>(a.num_q_tokens) * ((a.num_q_heads + hpc - 1) / hpc) : 0;
  const int64_t blocks = static_cast<int64_t>(a.num_tokens) + q_blocks;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dt == PHOTON_BF16)
    return launch_pdl(kv_cache_write_kernel<BF16Tag>, grid, dim3(kWriteThreads), 0, st, a, err);
  return launch_pdl(kv_cache_write_kernel<F32Tag>, grid, dim3(kWriteThreads), 0, st, a, err);
}

}  // namespace photon
