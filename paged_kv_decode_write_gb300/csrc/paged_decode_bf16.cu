// bf16-storage instantiations of the split-K paged decode kernels: the
// tensor-core kernel for head_dim 64 and 128, the CUDA-core kernel for
// head_dim 32 and 256 (query heads per KV head 1/2/4/8 throughout).
#include "paged_decode.cuh"
#include "paged_decode_mma.cuh"

namespace photon {

EncodeTiledFn tensor_map_encoder() {
  // looked up once (thread-safe initialisation of a function-local static)
  static const EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

cudaError_t launch_decode_partial_bf16(const DecodeArgs &a, unsigned int *err, cudaStream_t st) {
  // TMA row coordinates are 32-bit: the pool must have < 2^31 rows of head_dim
  const bool rows_fit = a.num_blocks * a.num_kv_heads * kBlockSize <= INT32_MAX;
  switch (a.head_dim) {
    case 32: return dispatch_group<BF16Tag, 32>(a, err, st);
    case 64:
      return rows_fit ? dispatch_mma_group<64>(a, err, st) : dispatch_group<BF16Tag, 64>(a, err, st);
    case 128:
      return rows_fit ? dispatch_mma_group<128>(a, err, st) : dispatch_group<BF16Tag, 128>(a, err, st);
    case 256: return dispatch_group<BF16Tag, 256>(a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
