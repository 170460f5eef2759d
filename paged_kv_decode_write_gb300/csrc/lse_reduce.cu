// Log-sum-exp merge of split-K partials (one warp per sequence x query head).
#include "paged_decode.cuh"

namespace photon {

cudaError_t launch_decode_reduce(const DecodeArgs &a, cudaStream_t st) {
  const int64_t warps = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  if (warps == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((warps + 7) / 8);
  switch (a.head_dim) {
    case 32: lse_reduce_kernel<32><<<grid, 256, 0, st>>>(a); break;
    case 64: lse_reduce_kernel<64><<<grid, 256, 0, st>>>(a); break;
    case 128: lse_reduce_kernel<128><<<grid, 256, 0, st>>>(a); break;
    case 256: lse_reduce_kernel<256><<<grid, 256, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace photon
