// Decode attention over a block-paged cache: the same kernels as the
// contiguous layout, instantiated with the block-table lookup in the group
// fetch (decode_kernel.cuh).  A separate translation unit so that the two
// instantiation sets compile in parallel.
#include "decode_kernel.cuh"

namespace kvq {

cudaError_t launch_paged(const DecodeArgs &a, int gq, cudaStream_t stream) {
  return a.geo.bits == 2 ? launch_b<2, true, false, false>(a, gq, stream) : launch_b<4, true, false, false>(a, gq, stream);
}

}  // namespace kvq
