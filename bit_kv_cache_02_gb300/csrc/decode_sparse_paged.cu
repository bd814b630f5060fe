// Decode attention over a block-paged cache of dense-and-sparse blocks
// (decode_sparse.cu with the block-table fetch).
#include "decode_kernel.cuh"

namespace kvq {

cudaError_t launch_sparse_paged(const DecodeArgs &a, int gq, cudaStream_t stream) {
  return a.geo.bits == 2 ? launch_b<2, true, false, true>(a, gq, stream) : launch_b<4, true, false, true>(a, gq, stream);
}

}  // namespace kvq
