// Batched KV-cache write with fused RoPE (sm_103a).
//
// PhotonInfer README, "Technical details > Paged attention": one kernel
// writes K/V for many sequences; "Key features > GPU-optimised kernels":
// batched RoPE as a fused operation.
//
// One CTA per written token.  Its threads first compute the token's rotation
// angles pos * theta^(-2i/d) in fp64, reduce them to [-pi, pi] and take
// sine and cosine once per pair (fp64, kept in shared memory); then they
// rotate that pair in every KV head (fp64 products, one round-to-nearest-even
// into the cache type) and copy the V rows with 16-byte vectors.  Rounding
// once from fp64 keeps the stored K within one unit in the last place of the
// exactly rotated value, whatever the cancellation in x*cos - y*sin.
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

template <typename Tag>
struct Store;
template <>
struct Store<F32Tag> {
  __device__ __forceinline__ static double load(const float *p, int64_t i) { return p[i]; }
  __device__ __forceinline__ static void put(float *p, int64_t i, double x) {
    p[i] = __double2float_rn(x);
  }
};
template <>
struct Store<BF16Tag> {
  __device__ __forceinline__ static double load(const __nv_bfloat16 *p, int64_t i) {
    return static_cast<double>(__bfloat162float(p[i]));
  }
  __device__ __forceinline__ static void put(__nv_bfloat16 *p, int64_t i, double x) {
    p[i] = f64_to_bf16(x);
  }
};

constexpr int kWriteThreads = 64;
constexpr int kMaxFp8Heads = 64;  // KV heads of an FP8 write (per-head scales in shared memory)

// cos / sin of pos * inv_freq[i] for the pairs of one position, into cs.
__device__ __forceinline__ void rope_table(const WriteArgs &a, int pos, double (*cs)[2]) {
  const double p = static_cast<double>(pos);
  for (int i = threadIdx.x; i < a.head_dim / 2; i += blockDim.x) {
    const double ang = p * a.inv_freq[i];
    const double k = rint(ang * kInvTwoPi);
    const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, ang));
    double s, c;
    sincos(r, &s, &c);
    cs[i][0] = c;
    cs[i][1] = s;
  }
  __syncthreads();
}

// Query heads one CTA rotates: as many as its threads cover pair by pair.
__host__ __device__ __forceinline__ int q_heads_per_cta(int head_dim) {
  const int h = kWriteThreads / (head_dim / 2);
  return h > 0 ? h : 1;
}

// Rotates heads [h0, h0 + q_heads_per_cta) of query row `row`
// ([num_q_heads][head_dim]) in place at q_positions[row].
template <typename Tag>
__device__ __forceinline__ void rotate_q_part(const WriteArgs &a, int row, int h0,
                                              double (*cs)[2]) {
  using T = typename Tag::T;
  if (a.rope_style == PHOTON_ROPE_NONE) return;
  rope_table(a, a.q_positions[row], cs);
  const int D = a.head_dim, half = D / 2;
  const int h1 = min(a.num_q_heads, h0 + q_heads_per_cta(D));
  const bool gptj = a.rope_style == PHOTON_ROPE_GPTJ;
  T *q = static_cast<T *>(a.q) + static_cast<int64_t>(row) * a.num_q_heads * D;
  for (int idx = h0 * half + threadIdx.x; idx < h1 * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const int e0 = gptj ? 2 * i : i;
    const int e1 = gptj ? 2 * i + 1 : i + half;
    const double x0 = Store<Tag>::load(q, h * D + e0);
    const double x1 = Store<Tag>::load(q, h * D + e1);
    Store<Tag>::put(q, h * D + e0, x0 * cs[i][0] - x1 * cs[i][1]);
    Store<Tag>::put(q, h * D + e1, x1 * cs[i][0] + x0 * cs[i][1]);
  }
}

template <typename Tag>
__global__ void __launch_bounds__(kWriteThreads)
    kv_cache_write_kernel(const __grid_constant__ WriteArgs a, unsigned int *err) {
  using T = typename Tag::T;
  __shared__ double cs[kMaxRopePairs][2];
  pdl_launch_dependents();
  pdl_wait();
  if (static_cast<int>(blockIdx.x) >= a.num_tokens) {  // part of a query row: rotate in place
    const int hpc = q_heads_per_cta(a.head_dim);
    const int per_row = (a.num_q_heads + hpc - 1) / hpc;
    const int qb = blockIdx.x - a.num_tokens;
    rotate_q_part<Tag>(a, qb / per_row, (qb % per_row) * hpc, cs);
    return;
  }
  const int64_t t = blockIdx.x;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (threadIdx.x == 0) atomicOr(err, PHOTON_DEVERR_SLOT_RANGE);
    return;
  }
  const int D = a.head_dim, half = D / 2, H = a.num_kv_heads;
  const int64_t blk = slot / kBlockSize, off = slot - blk * kBlockSize;

  // V: bit copy of each head row, 16 bytes at a time
  {
    constexpr int E = 16 / sizeof(T);
    const int per_row = D / E;
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.v) + t * H * D);
    T *vc = static_cast<T *>(a.v_cache);
    for (int idx = threadIdx.x; idx < H * per_row; idx += blockDim.x) {
      const int h = idx / per_row, ch = idx - h * per_row;
      uint4 *dst = reinterpret_cast<uint4 *>(vc + ((blk * H + h) * kBlockSize + off) * D);
      dst[ch] = src[h * per_row + ch];
    }
  }

  // K: sine / cosine of each pair's angle, once per token
  if (a.rope_style != PHOTON_ROPE_NONE) rope_table(a, a.positions[t], cs);
  const T *k = static_cast<const T *>(a.k) + t * H * D;
  T *kc = static_cast<T *>(a.k_cache);
  const bool gptj = a.rope_style == PHOTON_ROPE_GPTJ;
  const bool rotate = a.rope_style != PHOTON_ROPE_NONE;
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const int e0 = gptj ? 2 * i : i;
    const int e1 = gptj ? 2 * i + 1 : i + half;
    const int64_t dst = ((blk * H + h) * kBlockSize + off) * D;
    const double x0 = Store<Tag>::load(k, h * D + e0);
    const double x1 = Store<Tag>::load(k, h * D + e1);
    const double c = rotate ? cs[i][0] : 1.0, s = rotate ? cs[i][1] : 0.0;
    Store<Tag>::put(kc, dst + e0, x0 * c - x1 * s);
    Store<Tag>::put(kc, dst + e1, x1 * c + x0 * s);
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

// FP8 cache write: K pool [blocks][H_kv][bs][d] and V pool [blocks][H_kv][d][bs]
// of E4M3 codes; code = round(x * (1 / scale[h])) from the fp64 value x (RoPE'd
// for K), with the reciprocal taken in fp64.
template <typename Tag>
__global__ void __launch_bounds__(kWriteThreads)
    kv_cache_write_fp8_kernel(const __grid_constant__ WriteArgs a, const float *k_scale,
                              const float *v_scale, unsigned int *err) {
  using T = typename Tag::T;
  __shared__ double cs[kMaxRopePairs][2];
  __shared__ double inv_scale[2][kMaxFp8Heads];  // 1 / k_scale[h], 1 / v_scale[h] in fp64
  pdl_launch_dependents();
  pdl_wait();
  const int64_t t = blockIdx.x;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (threadIdx.x == 0) atomicOr(err, PHOTON_DEVERR_SLOT_RANGE);
    return;
  }
  const int D = a.head_dim, half = D / 2, H = a.num_kv_heads;
  const int64_t blk = slot / kBlockSize, off = slot - blk * kBlockSize;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    inv_scale[0][h] = 1.0 / static_cast<double>(k_scale[h]);
    inv_scale[1][h] = 1.0 / static_cast<double>(v_scale[h]);
  }
  __syncthreads();
  const T *v = static_cast<const T *>(a.v) + t * H * D;
  unsigned char *vc = static_cast<unsigned char *>(a.v_cache);
  for (int idx = threadIdx.x; idx < H * D; idx += blockDim.x) {
    const int h = idx / D, e = idx - h * D;
    const double y = Store<Tag>::load(v, idx) * inv_scale[1][h];
    vc[((blk * H + h) * D + e) * kBlockSize + off] = f64_to_e4m3(y);
  }
  const bool rotate = a.rope_style != PHOTON_ROPE_NONE;
  if (rotate) rope_table(a, a.positions[t], cs);
  const T *k = static_cast<const T *>(a.k) + t * H * D;
  unsigned char *kc = static_cast<unsigned char *>(a.k_cache);
  const bool gptj = a.rope_style == PHOTON_ROPE_GPTJ;
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const int e0 = gptj ? 2 * i : i;
    const int e1 = gptj ? 2 * i + 1 : i + half;
    const int64_t dst = ((blk * H + h) * kBlockSize + off) * D;
    const double x0 = Store<Tag>::load(k, h * D + e0);
    const double x1 = Store<Tag>::load(k, h * D + e1);
    const double c = rotate ? cs[i][0] : 1.0, s = rotate ? cs[i][1] : 0.0;
    kc[dst + e0] = f64_to_e4m3((x0 * c - x1 * s) * inv_scale[0][h]);
    kc[dst + e1] = f64_to_e4m3((x1 * c + x0 * s) * inv_scale[0][h]);
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
