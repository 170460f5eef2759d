// Batched KV-cache write with fused RoPE (sm_103a).
//
// PhotonInfer README, "Technical details > Paged attention": one kernel
// writes K/V for many sequences; "Key features > GPU-optimised kernels":
// batched RoPE as a fused operation.  Each thread owns one rotation pair i of
// one token: it computes the angle and its sine/cosine once in fp64 and
// applies them to that pair in every KV head, then stores the rotated K
// (rounded once to nearest-even) and the unrotated V at the token's slot.
// Loads and stores of a warp cover consecutive elements of one head row, so
// they coalesce; the kernel is tiny next to the attention read.
#include "common.cuh"
#include "internal.h"

namespace photon {
namespace {

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

template <typename Tag>
__global__ void __launch_bounds__(128) kv_cache_write_kernel(const WriteArgs a, unsigned int *err) {
  using T = typename Tag::T;
  const int half = a.head_dim / 2;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t t = idx / half;
  const int i = static_cast<int>(idx - t * half);
  if (t >= a.num_tokens) return;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= a.num_slots) {
    if (i == 0) atomicOr(err, PHOTON_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / kBlockSize, off = slot - blk * kBlockSize;
  const int e0 = a.rope_style == PHOTON_ROPE_GPTJ ? 2 * i : i;
  const int e1 = a.rope_style == PHOTON_ROPE_GPTJ ? 2 * i + 1 : i + half;
  double c = 1.0, s = 0.0;
  if (a.rope_style != PHOTON_ROPE_NONE) {
    const double ang = static_cast<double>(a.positions[t]) * a.inv_freq[i];
    sincos(ang, &s, &c);
  }
  const T *k = static_cast<const T *>(a.k);
  const T *v = static_cast<const T *>(a.v);
  T *kc = static_cast<T *>(a.k_cache);
  T *vc = static_cast<T *>(a.v_cache);
  for (int h = 0; h < a.num_kv_heads; ++h) {
    const int64_t src = (t * a.num_kv_heads + h) * a.head_dim;
    const int64_t dst = ((blk * a.num_kv_heads + h) * kBlockSize + off) * a.head_dim;
    const double x0 = Store<Tag>::load(k, src + e0);
    const double x1 = Store<Tag>::load(k, src + e1);
    Store<Tag>::put(kc, dst + e0, x0 * c - x1 * s);
    Store<Tag>::put(kc, dst + e1, x1 * c + x0 * s);
    vc[dst + e0] = v[src + e0];
    vc[dst + e1] = v[src + e1];
  }
}

}  // namespace

cudaError_t launch_kv_cache_write(const WriteArgs &a, photon_dtype dt, unsigned int *err,
                                  cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a.num_tokens) * (a.head_dim / 2);
  if (threads == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((threads + 127) / 128);
  if (dt == PHOTON_BF16)
    kv_cache_write_kernel<BF16Tag><<<grid, 128, 0, st>>>(a, err);
  else
    kv_cache_write_kernel<F32Tag><<<grid, 128, 0, st>>>(a, err);
  return cudaGetLastError();
}

}  // namespace photon
