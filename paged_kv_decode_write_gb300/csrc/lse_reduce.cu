// Log-sum-exp merge of split-K partials (one warp per sequence x query head).
#include "paged_decode.cuh"

namespace photon {

cudaError_t launch_decode_reduce(const DecodeArgs &a, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  if (rows == 0) return cudaSuccess;
  if (rows > INT32_MAX) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(rows));
  switch (a.head_dim) {
    case 32: return launch_pdl(lse_reduce_kernel<32>, grid, dim3(ReduceCfg<32>::THREADS), 0, st, a);
    case 64: return launch_pdl(lse_reduce_kernel<64>, grid, dim3(ReduceCfg<64>::THREADS), 0, st, a);
    case 128: return launch_pdl(lse_reduce_kernel<128>, grid, dim3(ReduceCfg<128>::THREADS), 0, st, a);
    case 256: return launch_pdl(lse_reduce_kernel<256>, grid, dim3(ReduceCfg<256>::THREADS), 0, st, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace photon
