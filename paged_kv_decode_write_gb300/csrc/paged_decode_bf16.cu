// bf16-storage instantiations of the split-K paged decode kernel
// (head_dim 32/64/128/256 x query heads per KV head 1/2/4/8).
#include "paged_decode.cuh"

namespace photon {

cudaError_t launch_decode_partial_bf16(const DecodeArgs &a, unsigned int *err, cudaStream_t st) {
  switch (a.head_dim) {
    case 32: return dispatch_group<BF16Tag, 32>(a, err, st);
    case 64: return dispatch_group<BF16Tag, 64>(a, err, st);
    case 128: return dispatch_group<BF16Tag, 128>(a, err, st);
    case 256: return dispatch_group<BF16Tag, 256>(a, err, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
